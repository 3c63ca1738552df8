"""MXFP8 microscaled quantization and block-scaled FP8 GEMMs for GB300 (sm_103a).

The compute runs in the CUDA library ``libmxq.so`` built from ``csrc/``; the
Python layer (``mxq``) only marshals arguments through its C ABI.  Importing
the package does not load the library; the first call does, and raises if the
library has not been built.
"""

__all__ = ["mxq", "workloads"]
