#!/usr/bin/env python3
"""Benchmark of the MXFP8 training hot path on GB300.

One step = one pass of the hot path over one batch of synthetic input.  The
default workload is the largest single-GPU linear layer, M = 16384 tokens,
K = N = 16384 (activations 0.5 Student-t(3), weights N(0, 0.02^2)): dual-axis
1x32 quantization of X, W and dY, then the forward (Y = X W^T), dgrad
(dX = dY W) and wgrad (dW = dY^T X) block-scaled GEMMs with BF16 output.
The same process then times the 128-expert MoE grouped GEMMs (16384 tokens,
top-8, gate_up and down projections with their row quantizations) and adds
them under `moe_block` (--extra-workloads).  Other workloads (--workload):
linear_train (8192 x 4096 x 4096), linear_fwd_small, weight_32x32 (32x32
weight payload shared by forward and dgrad), moe_grouped, moe_train,
fsdp_*, sweep_4096 / sweep_7168.

Prints one JSON line.  `value` is the step's GEMM FLOPs divided by the step
time (quantizers included), inputs resident in HBM, timed with CUDA events
on the launching stream; L2 is flushed (256 MB write) between timed steps,
outside the timed intervals.  `e2e` is the same metric through the public
API with the inputs copied from pinned host memory and the BF16 results
copied back inside every timed step.  `roofline` covers the GEMM kernel
(peak: the larger of 2 x the measured BF16 burst and the vendor library's
MXFP8 GEMM timed in the same run), `roofline_quant` the quantizers.
`cpu_baseline` times the oracle on a bounded sample.  `--impl reference`
times the oracle alone (CPU).

Multi-GPU: the path has no exchange step, so N ranks run N independent
replicas (weak scaling); the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
# Step entries that launch more than one kernel of the library.
LAUNCHES_PER_ENTRY = {"quant_XW_dual": 2}

if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MXFP8 GEMM TFLOP/s (% dense MXFP8 peak); quantizer TB/s (% HBM), 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0          # nominal dense ratio (4.5 / 2.25 PFLOP/s)
L2_FLUSH_BYTES = 256 << 20   # larger than the 129 MB L2
L2_BYTES = 129 * 10**6
# DRAM bytes (read + write) per GEMM launch of one step, averaged over the step's
# GEMM launches like `units_per_launch`, from an ncu capture of the kernel as it
# stands; None where not captured (or captured before the kernel last changed).
GEMM_TRAFFIC_BYTES = {
    # gemm_mxf8_pair_kernel as it stands (ncu dram__bytes_read/write.sum, the second step's
    # launches).  sweep_16384 runs on clusters of two pairs <0,0,4>: forward 3.664 GB read +
    # 0.530 GB written, dgrad + wgrad 7.218 + 1.064 GB
    "sweep_16384": int((3.664e9 + 0.530e9 + 7.218e9 + 1.064e9) / 2),
    # 8192x4096x4096 on single pairs <0,0,2>: forward 51.97 + 33.52 MB, dgrad + wgrad 137.01 + 65.23 MB
    "linear_train": int((51.97e6 + 33.52e6 + 137.01e6 + 65.23e6) / 2),
}
DEFAULT_WORKLOAD = "sweep_16384"
DEFAULT_EXTRA = "moe_grouped"
# Shapes (M, N, K) at which the vendor library's MXFP8 GEMM is timed for the
# GEMM peak: its best measured rate on this machine, next to the workload's own.
VENDOR_SHAPES = [(8192, 4096, 4096), (16384, 8192, 8192), (16384, 16384, 16384)]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


# ---- distributed plumbing (replicas; only timing crosses ranks) ------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate_value(flops_per_rank_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job TFLOP/s: the FLOPs all ranks did divided by the slowest rank's time."""
    return flops_per_rank_step * steps * world / max_seconds / 1e12


# ---- clocks -----------------------------------------------------------------------------

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = [p for (t, p) in self.samples if t0 <= t <= t1] or [p for (_, p) in self.samples]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        capped = sum(1 for r in rows if r[8].lower().startswith("active"))
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "sm_mhz_min": min(sm) if sm else None, "sm_mhz_mean": round(statistics.mean(sm), 1) if sm else None,
                "power_w_max": max(pw) if pw else None, "power_cap_samples": capped,
                "reasons": reasons, "samples": len(rows)}


# ---- workloads -----------------------------------------------------------------------------

class Workload:
    """Device tensors, preallocated outputs and the ordered kernel launches of one step."""
    name = ""
    inputs: dict
    outputs: list
    state_keys = ()   # inputs that are model state (weights): resident in HBM, not copied per step

    def kernels(self):
        """[(name, kind, algorithmic units, launch fn)]: kind 'gemm' (units = FLOPs)
        or 'quant' (units = bytes moved by the algorithm)."""
        raise NotImplementedError

    @property
    def gemm_flops(self):
        """GEMM FLOPs of one step (2 per multiply-add)."""
        raise NotImplementedError


def _dual_bytes(r, c):
    return r * c * (2 + 1 + 1) + 2 * (r * c // 32)


def _group_tiled_setup(w, offsets_cpu, ks, dev):
    """Group-tiled A-scale buffers of the routed rows for the grouped GEMMs (one
    per contraction length in ks), their band capacity and the bands the
    routing fills (each expert's rows ceil(n_g / 128) bands)."""
    import torch
    from mxfp8_microscaled_precision_gb300 import mxq
    off = [int(v) for v in offsets_cpu]
    w.gt_cap = mxq.group_tiled_bands(w.Mt, w.G)
    w.gt_bands = sum((hi - lo + 127) // 128 for lo, hi in zip(off[:-1], off[1:]) if hi > lo)
    return [torch.empty(w.gt_cap * (k // 128) * 512, dtype=torch.uint8, device=dev) for k in ks]


def _regroup_bytes(w, k):
    """Algorithmic bytes of one regroup: the tiled scales of all routed rows
    read once, the filled group-tiled bands written."""
    return ((w.Mt + 127) // 128 + w.gt_bands) * (k // 128) * 512


def _row_bytes(r, c):
    return r * c * (2 + 1) + r * c // 32


def _blk_bytes(r, c):
    return r * c * (2 + 1) + 2 * (r * c // 32)


class LinearTrain(Workload):
    state_keys = ("W",)

    def __init__(self, name, M, N, K, gen, dev=None):
        import torch
        from mxfp8_microscaled_precision_gb300 import mxq
        self.name, self.M, self.N, self.K = name, M, N, K
        self.inputs = gen(dev or "cpu")
        if dev is None:          # host-only: the oracle arm
            return
        u8 = dict(dtype=torch.uint8, device=dev)

        def dual_out(r, c):
            return (torch.empty((r, c), **u8), torch.empty(mxq.scale_bytes(r, c), **u8),
                    torch.empty((c, r), **u8), torch.empty(mxq.scale_bytes(c, r), **u8))
        self.qx, self.qw, self.qg = dual_out(M, K), dual_out(N, K), dual_out(M, N)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.y, self.dx, self.dw = torch.empty((M, N), **bf), torch.empty((M, K), **bf), torch.empty((N, K), **bf)
        self.outputs = [self.y, self.dx, self.dw]
        gr, grs, gc, gcs = self.qg
        # X and W are quantized on two streams: the second kernel's CTAs take the
        # SM slots the first one frees in its last, partly filled round
        self.side = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
        self.bwd = [dict(a_q=gr, a_s=grs, b_q=self.qw[2], b_s=self.qw[3], M=M, N=K, K=N, out=self.dx),
                    dict(a_q=gc, a_s=gcs, b_q=self.qx[2], b_s=self.qx[3], M=N, N=K, K=M, out=self.dw)]

    @property
    def gemm_flops(self):
        return 3 * 2 * self.M * self.N * self.K

    def kernels(self):
        from mxfp8_microscaled_precision_gb300 import mxq
        M, N, K, i = self.M, self.N, self.K, self.inputs
        xr, xrs, xc, xcs = self.qx
        wr, wrs, wc, wcs = self.qw
        gr, grs, gc, gcs = self.qg
        return [
            ("quant_XW_dual", "quant", _dual_bytes(M, K) + _dual_bytes(N, K), self._quant_xw),
            ("quant_dY_dual", "quant", _dual_bytes(M, N), lambda: mxq.quant_1x32_dual(i["dY"], out=self.qg)),
            ("gemm_fwd", "gemm", 2 * M * N * K, lambda: mxq.gemm(xr, xrs, wr, wrs, M, N, K, out=self.y)),
            # dgrad dX = dY W and wgrad dW = dY^T X share one launch (one last wave of tiles)
            ("gemm_bwd", "gemm", 2 * 2 * M * N * K, lambda: mxq.gemm_multi(self.bwd)),
        ]

    def _quant_xw(self):
        import torch
        from mxfp8_microscaled_precision_gb300 import mxq
        cur = torch.cuda.current_stream()
        for s in self.side:
            s.wait_stream(cur)
        with torch.cuda.stream(self.side[0]):
            mxq.quant_1x32_dual(self.inputs["X"], out=self.qx)
        with torch.cuda.stream(self.side[1]):
            mxq.quant_1x32_dual(self.inputs["W"], out=self.qw)
        for s in self.side:
            cur.wait_stream(s)

    def cpu_sample(self, budget_s):
        """Times the oracle on a bounded sample of each step part: the dual
        quantization of 256 rows of X, and FP64 GEMM output rows against the
        first 512 rows of W (output columns), one row at a time until the budget.
        Returns (seconds per full step extrapolated from those rates, description)."""
        from oracle import oracle
        import numpy as np
        i = self.inputs
        x = _host_bits(i["X"][:256])
        t0 = time.perf_counter()
        oracle.quant_dual(x)
        tq = (time.perf_counter() - t0) / x.size          # per element, dual
        qr, sr = oracle.quant_rows(_host_bits(i["X"][:64]))
        a = oracle.dequant_rows(qr, sr)
        ncols = min(512, self.N)
        wq, ws = oracle.quant_rows(_host_bits(i["W"][:ncols]))
        b = oracle.dequant_rows(wq, ws)
        rows, t_g = 0, 0.0
        while t_g < budget_s and rows < a.shape[0]:
            t0 = time.perf_counter()
            oracle.gemm(a, b, rows=np.array([rows], dtype=np.int64))
            t_g += time.perf_counter() - t0
            rows += 1
        tg = t_g / (2.0 * rows * ncols * self.K)          # per FLOP
        quant_elems = self.M * self.K + self.N * self.K + self.M * self.N
        step = tq * quant_elems + tg * self.gemm_flops
        return step, (f"oracle dual quant of 256 rows of X ({x.size} elements) and FP64 GEMM of "
                      f"{rows} output rows x {ncols} output columns x K {self.K}; rates extrapolated to the "
                      f"full step ({quant_elems} quantized elements, {self.gemm_flops:.4g} GEMM FLOPs)")


class LinearFwdSmall(Workload):
    state_keys = ("W",)

    def __init__(self, dev=None):
        import torch
        from mxfp8_microscaled_precision_gb300 import mxq, workloads
        self.name, self.M, self.N, self.K = "linear_fwd_small", 256, 512, 512
        self.inputs = workloads.linear_fwd_small(dev or "cpu")
        if dev is None:
            return
        u8 = dict(dtype=torch.uint8, device=dev)
        self.qx = (torch.empty((256, 512), **u8), torch.empty(mxq.scale_bytes(256, 512), **u8), None, None)
        self.qw = (torch.empty((512, 512), **u8), torch.empty(mxq.scale_bytes(512, 512), **u8), None, None)
        self.y = torch.empty((256, 512), dtype=torch.bfloat16, device=dev)
        self.outputs = [self.y]

    @property
    def gemm_flops(self):
        return 2 * self.M * self.N * self.K

    def kernels(self):
        from mxfp8_microscaled_precision_gb300 import mxq
        i = self.inputs
        return [
            ("quant_X_row", "quant", _row_bytes(256, 512), lambda: mxq.quant_1x32_dual(i["X"], col=False, out=self.qx)),
            ("quant_W_row", "quant", _row_bytes(512, 512), lambda: mxq.quant_1x32_dual(i["W"], col=False, out=self.qw)),
            ("gemm_fwd", "gemm", 2 * 256 * 512 * 512,
             lambda: mxq.gemm(self.qx[0], self.qx[1], self.qw[0], self.qw[1], 256, 512, 512, out=self.y)),
        ]

    def cpu_sample(self, budget_s):
        from oracle import oracle
        i = self.inputs
        t0 = time.perf_counter()
        xq, xs = oracle.quant_rows(_host_bits(i["X"]))
        wq, ws = oracle.quant_rows(_host_bits(i["W"]))
        oracle.gemm(oracle.dequant_rows(xq, xs), oracle.dequant_rows(wq, ws))
        return time.perf_counter() - t0, "the whole step (quantization of X and W, FP64 GEMM)"


class LinearFwdChain(Workload):
    """Forward of one linear layer whose output feeds the next MXFP8 layer:
    Y = X W^T in BF16 plus Y's 1x32 row quantization (the next layer's input),
    either from the GEMM's quantizing epilogue ("fused") or by a separate
    quantizer pass over Y ("two_pass").  Shapes of linear_train."""
    state_keys = ("W",)

    def __init__(self, fused, dev=None, M=8192, N=4096, K=4096):
        import torch
        from mxfp8_microscaled_precision_gb300 import mxq, workloads
        self.fused = fused
        self.name = "linear_fwd_chain_" + ("fused" if fused else "two_pass")
        self.M, self.N, self.K = M, N, K
        d = workloads.linear_train(dev or "cpu", M, N, K)
        self.inputs = {"X": d["X"], "W": d["W"]}
        if dev is None:
            return
        u8 = dict(dtype=torch.uint8, device=dev)
        self.qx = (torch.empty((M, K), **u8), torch.empty(mxq.scale_bytes(M, K), **u8), None, None)
        self.qw = (torch.empty((N, K), **u8), torch.empty(mxq.scale_bytes(N, K), **u8), None, None)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.qy = (torch.empty((M, N), **u8), torch.empty(mxq.scale_bytes(M, N), **u8), None, None)
        self.outputs = [self.y, self.qy[0], self.qy[1]]

    @property
    def gemm_flops(self):
        return 2 * self.M * self.N * self.K

    def kernels(self):
        from mxfp8_microscaled_precision_gb300 import mxq
        M, N, K, i = self.M, self.N, self.K, self.inputs
        ks = [("quant_X_row", "quant", _row_bytes(M, K), lambda: mxq.quant_1x32_dual(i["X"], col=False, out=self.qx)),
              ("quant_W_row", "quant", _row_bytes(N, K), lambda: mxq.quant_1x32_dual(i["W"], col=False, out=self.qw))]
        if self.fused:
            ks.append(("gemm_fwd_quantout", "gemm", 2 * M * N * K,
                       lambda: mxq.gemm_mxfp8out(self.qx[0], self.qx[1], self.qw[0], self.qw[1], M, N, K,
                                                 out=(self.y, self.qy[0], self.qy[1]))))
        else:
            ks.append(("gemm_fwd", "gemm", 2 * M * N * K,
                       lambda: mxq.gemm(self.qx[0], self.qx[1], self.qw[0], self.qw[1], M, N, K, out=self.y)))
            ks.append(("quant_Y_row", "quant", _row_bytes(M, N),
                       lambda: mxq.quant_1x32_dual(self.y, col=False, out=self.qy)))
        return ks

    def cpu_sample(self, budget_s):
        from oracle import oracle
        import numpy as np
        i = self.inputs
        x = _host_bits(i["X"][:64])
        t0 = time.perf_counter()
        xq, xs = oracle.quant_rows(x)
        tq = (time.perf_counter() - t0) / x.size
        a = oracle.dequant_rows(xq, xs)
        wq, ws = oracle.quant_rows(_host_bits(i["W"]))
        b = oracle.dequant_rows(wq, ws)
        rows, t_g = 0, 0.0
        while t_g < budget_s and rows < a.shape[0]:
            t0 = time.perf_counter()
            y = oracle.gemm(a, b, rows=np.array([rows], dtype=np.int64))
            oracle.quant_rows(y.reshape(1, -1))
            t_g += time.perf_counter() - t0
            rows += 1
        tg = t_g / (2.0 * rows * self.N * self.K)
        elems = self.M * self.K + self.N * self.K
        return tq * elems + tg * self.gemm_flops, (
            f"oracle row quant of 64 rows of X and FP64 GEMM + row quant of {rows} output rows x {self.N} x "
            f"{self.K}; extrapolated to the full step")


class Weight32(Workload):
    state_keys = ("W",)

    def __init__(self, dev=None):
        import torch
        from mxfp8_microscaled_precision_gb300 import mxq, workloads
        self.name, self.M, self.n, self.k = "weight_32x32", 4096, 7168, 7168
        self.inputs = workloads.weight_32x32(dev or "cpu")
        if dev is None:
            return
        M, n, k = self.M, self.n, self.k
        u8 = dict(dtype=torch.uint8, device=dev)
        self.qw = (torch.empty((n, k), **u8), torch.empty(mxq.scale_bytes(n, k), **u8),
                   torch.empty(mxq.scale_bytes(k, n), **u8))
        self.qx = (torch.empty((M, k), **u8), torch.empty(mxq.scale_bytes(M, k), **u8), None, None)
        self.qg = (torch.empty((M, n), **u8), torch.empty(mxq.scale_bytes(M, n), **u8), None, None)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.y, self.dx = torch.empty((M, n), **bf), torch.empty((M, k), **bf)
        self.outputs = [self.y, self.dx]

    @property
    def gemm_flops(self):
        return 2 * 2 * self.M * self.n * self.k

    def kernels(self):
        from mxfp8_microscaled_precision_gb300 import mxq
        M, n, k, i = self.M, self.n, self.k, self.inputs
        q, sf, sb = self.qw
        return [
            ("quant_W_32x32", "quant", _blk_bytes(n, k), lambda: mxq.quant_32x32(i["W"], out=self.qw)),
            ("quant_X_row", "quant", _row_bytes(M, k), lambda: mxq.quant_1x32_dual(i["X"], col=False, out=self.qx)),
            ("quant_dY_row", "quant", _row_bytes(M, n), lambda: mxq.quant_1x32_dual(i["dY"], col=False, out=self.qg)),
            ("gemm_fwd", "gemm", 2 * M * n * k, lambda: mxq.gemm(self.qx[0], self.qx[1], q, sf, M, n, k, out=self.y)),
            ("gemm_dgrad_mn", "gemm", 2 * M * n * k,
             lambda: mxq.gemm(self.qg[0], self.qg[1], q, sb, M, k, n, b_mn_major=True, out=self.dx)),
        ]

    def cpu_sample(self, budget_s):
        from oracle import oracle
        import numpy as np
        i = self.inputs
        w = _host_bits(i["W"][:256])
        t0 = time.perf_counter()
        oracle.quant_32x32(w)
        tq = (time.perf_counter() - t0) / w.size
        xq, xs = oracle.quant_rows(_host_bits(i["X"][:64]))
        a = oracle.dequant_rows(xq, xs)
        oq, osf, _ = oracle.quant_32x32(_host_bits(i["W"]))
        b = oracle.dequant_rows(oq, osf)
        rows, t_g = 0, 0.0
        while t_g < budget_s and rows < a.shape[0]:
            t0 = time.perf_counter()
            oracle.gemm(a, b, rows=np.array([rows], dtype=np.int64))
            t_g += time.perf_counter() - t0
            rows += 1
        tg = t_g / (2.0 * rows * self.n * self.k)
        elems = self.n * self.k + self.M * self.k + self.M * self.n
        return tq * elems + tg * self.gemm_flops, (
            f"oracle 32x32 quant of 256 weight rows and FP64 GEMM of {rows} rows x {self.n} x {self.k}; "
            f"extrapolated to the full step")


class FsdpWeight(Workload):
    """One fully sharded linear layer seen from rank 0 of `world` ranks (MindSpeed
    RFC "Add MXFP8-32x32 quantization support to FSDP", section 3.3.2): quantize
    the local weight shard straight into its all-gather payload, receive the other
    ranks' payloads (device copies stand in for the collective on one GPU), rebuild
    the full operands, then the forward and dgrad GEMMs of the 7168x7168 layer
    with X and dY [4096, 7168] row-quantized.  recipe "mxfp8" gathers four tensors
    per rank, "mxfp8-32x32" three."""

    state_keys = ("W_shard",)

    def __init__(self, recipe, dev=None, world=8):
        import torch
        from mxfp8_microscaled_precision_gb300 import mxq, workloads
        self.recipe = recipe
        self.name = "fsdp_" + recipe.replace("-", "_")
        self.M, self.n, self.k, self.world = 4096, 7168, 7168, world
        ns = self.n // world
        d = workloads.weight_32x32(dev or "cpu")
        self.inputs = {"W_shard": d["W"][:ns].contiguous(), "X": d["X"], "dY": d["dY"]}
        if dev is None:
            return
        M, n, k = self.M, self.n, self.k
        u8 = dict(dtype=torch.uint8, device=dev)
        self.off, self.P = mxq.fsdp_payload_layout(recipe, n, k, world)
        self.gathered = torch.zeros(world * self.P, **u8)
        self.remote = torch.zeros((world - 1) * self.P, **u8)     # the other ranks' send buffers
        for r in range(1, world):
            mxq.fsdp_quant_shard(d["W"][r * ns:(r + 1) * ns], recipe, n, world,
                                 self.remote[(r - 1) * self.P:r * self.P])
        del d["W"]
        dual = recipe == "mxfp8"
        self.full = (torch.empty((n, k), **u8), torch.empty(mxq.scale_bytes(n, k), **u8),
                     torch.empty((k, n), **u8) if dual else None, torch.empty(mxq.scale_bytes(k, n), **u8))
        self.qx = (torch.empty((M, k), **u8), torch.empty(mxq.scale_bytes(M, k), **u8), None, None)
        self.qg = (torch.empty((M, n), **u8), torch.empty(mxq.scale_bytes(M, n), **u8), None, None)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.y, self.dx = torch.empty((M, n), **bf), torch.empty((M, k), **bf)
        self.outputs = [self.y, self.dx]
        torch.cuda.synchronize()

    @property
    def gemm_flops(self):
        return 2 * 2 * self.M * self.n * self.k

    def extra(self):
        n, k, W, P = self.n, self.k, self.world, self.P
        return {"fsdp": {"recipe": self.recipe, "world": W, "tensors_per_rank": sum(o >= 0 for o in self.off),
                         "payload_bytes_per_rank": P, "gathered_bytes": W * P,
                         "bytes_per_weight_element": round(W * P / (n * k), 5),
                         "collective": "stood in for by one device copy of the other ranks' payloads"}}

    def kernels(self):
        from mxfp8_microscaled_precision_gb300 import mxq
        M, n, k, W, P, i = self.M, self.n, self.k, self.world, self.P, self.inputs
        ns = n // W
        q, sf, qc, sb = self.full
        dual = self.recipe == "mxfp8"
        own = self.gathered[:P]
        if dual:
            dgrad = ("gemm_dgrad", "gemm", 2 * M * n * k,
                     lambda: mxq.gemm(self.qg[0], self.qg[1], qc, sb, M, k, n, out=self.dx))
        else:
            dgrad = ("gemm_dgrad_mn", "gemm", 2 * M * n * k,
                     lambda: mxq.gemm(self.qg[0], self.qg[1], q, sb, M, k, n, b_mn_major=True, out=self.dx))
        return [
            ("quant_W_shard", "quant", _dual_bytes(ns, k) if dual else _blk_bytes(ns, k),
             lambda: mxq.fsdp_quant_shard(i["W_shard"], self.recipe, n, W, own)),
            ("allgather_copy", "collective", 2 * (W - 1) * P, lambda: self.gathered[P:].copy_(self.remote)),
            ("fsdp_unpack", "copy", 2 * W * P,
             lambda: mxq.fsdp_unpack(self.recipe, self.gathered, n, k, W, out=self.full)),
            ("quant_X_row", "quant", _row_bytes(M, k), lambda: mxq.quant_1x32_dual(i["X"], col=False, out=self.qx)),
            ("quant_dY_row", "quant", _row_bytes(M, n), lambda: mxq.quant_1x32_dual(i["dY"], col=False, out=self.qg)),
            ("gemm_fwd", "gemm", 2 * M * n * k, lambda: mxq.gemm(self.qx[0], self.qx[1], q, sf, M, n, k, out=self.y)),
            dgrad,
        ]

    def cpu_sample(self, budget_s):
        from oracle import oracle
        import numpy as np
        i = self.inputs
        w = _host_bits(i["W_shard"][:256])
        t0 = time.perf_counter()
        if self.recipe == "mxfp8":
            oracle.quant_dual(w)
        else:
            oracle.quant_32x32(w)
        tq = (time.perf_counter() - t0) / w.size
        xq, xs = oracle.quant_rows(_host_bits(i["X"][:64]))
        a = oracle.dequant_rows(xq, xs)
        # the GEMM rate from output rows against this rank's shard of W (its rows
        # are the weight's first n/world output features)
        w_shard = i["W_shard"]
        ns = w_shard.shape[0]
        wq, ws = oracle.quant_rows(_host_bits(w_shard))
        b = oracle.dequant_rows(wq, ws)
        rows, t_g = 0, 0.0
        while t_g < budget_s and rows < a.shape[0]:
            t0 = time.perf_counter()
            oracle.gemm(a, b, rows=np.array([rows], dtype=np.int64))
            t_g += time.perf_counter() - t0
            rows += 1
        tg = t_g / (2.0 * rows * ns * self.k)
        elems = self.n * self.k // self.world + self.M * self.k + self.M * self.n
        return tq * elems + tg * self.gemm_flops, (
            f"oracle {self.recipe} quant of 256 shard rows and FP64 GEMM of {rows} rows x {ns} x {self.k} "
            f"(the rank's shard of W); extrapolated to the full step (the gather and unpack move bytes only "
            f"and are not timed on the CPU)")


class MoE(Workload):
    state_keys = ("W_gate_up", "W_down")

    def __init__(self, dev=None):
        import torch
        from mxfp8_microscaled_precision_gb300 import mxq, workloads
        self.name = "moe_grouped"
        d = workloads.moe_grouped(dev or "cpu", weights=False)
        G, H, I = 128, 4096, 2048
        self.G, self.H, self.I = G, H, I
        self.Mt = d["A"].shape[0]
        seed_gu = workloads.seed_for("moe_grouped", "W")
        seed_dn = workloads.seed_for("moe_grouped", "W_down")
        if dev is None:          # host-only: the oracle arm needs one expert's weights
            self.inputs = {"A": d["A"], "Hd": d["H"],
                           "W_gate_up": workloads.normal((2 * I, H), 0.02, seed_gu)}
            return
        self.offsets = d["routing"].offsets.to(dev)
        self.inputs = {"A": d["A"], "Hd": d["H"], "offsets": self.offsets,
                       "W_gate_up": workloads.normal((G * 2 * I, H), 0.02, seed_gu, device=dev),
                       "W_down": workloads.normal((G * H, I), 0.02, seed_dn, device=dev)}
        u8 = dict(dtype=torch.uint8, device=dev)

        def row_out(r, c):
            return (torch.empty((r, c), **u8), torch.empty(mxq.scale_bytes(r, c), **u8), None, None)
        self.qa, self.qh = row_out(self.Mt, H), row_out(self.Mt, I)
        self.qgu, self.qdn = row_out(G * 2 * I, H), row_out(G * H, I)
        self.sa_g, self.sh_g = _group_tiled_setup(self, d["routing"].offsets, (H, I), dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.y1, self.y2 = torch.empty((self.Mt, 2 * I), **bf), torch.empty((self.Mt, H), **bf)
        self.outputs = [self.y1, self.y2]

    @property
    def gemm_flops(self):
        return 2 * self.Mt * 2 * self.I * self.H + 2 * self.Mt * self.H * self.I

    def kernels(self):
        from mxfp8_microscaled_precision_gb300 import mxq
        i, G, H, I, Mt = self.inputs, self.G, self.H, self.I, self.Mt
        return [
            ("quant_A_row", "quant", _row_bytes(Mt, H), lambda: mxq.quant_1x32_dual(i["A"], col=False, out=self.qa)),
            ("quant_H_row", "quant", _row_bytes(Mt, I), lambda: mxq.quant_1x32_dual(i["Hd"], col=False, out=self.qh)),
            ("regroup_A_scales", "layout", _regroup_bytes(self, H),
             lambda: mxq.scale_regroup_rows(self.qa[1], Mt, H, self.offsets, self.gt_cap, out=self.sa_g)),
            ("regroup_H_scales", "layout", _regroup_bytes(self, I),
             lambda: mxq.scale_regroup_rows(self.qh[1], Mt, I, self.offsets, self.gt_cap, out=self.sh_g)),
            ("quant_Wgu_row", "quant", _row_bytes(G * 2 * I, H),
             lambda: mxq.quant_1x32_dual(i["W_gate_up"], col=False, out=self.qgu)),
            ("quant_Wdn_row", "quant", _row_bytes(G * H, I),
             lambda: mxq.quant_1x32_dual(i["W_down"], col=False, out=self.qdn)),
            ("grouped_gate_up", "gemm", 2 * Mt * 2 * I * H,
             lambda: mxq.grouped_gemm_group_tiled(self.qa[0], self.sa_g, self.qgu[0], self.qgu[1], self.offsets,
                                                  2 * I, H, self.gt_cap, out=self.y1)),
            ("grouped_down", "gemm", 2 * Mt * H * I,
             lambda: mxq.grouped_gemm_group_tiled(self.qh[0], self.sh_g, self.qdn[0], self.qdn[1], self.offsets,
                                                  H, I, self.gt_cap, out=self.y2)),
        ]

    def expert0_gate_up(self):
        """Expert 0's gate_up weight [2I, H] (stacked rows on the device, alone on the host)."""
        return self.inputs["W_gate_up"][:2 * self.I]

    def cpu_sample(self, budget_s):
        from oracle import oracle
        import numpy as np
        i = self.inputs
        x = _host_bits(i["A"][:256])
        t0 = time.perf_counter()
        oracle.quant_rows(x)
        tq = (time.perf_counter() - t0) / x.size
        qa, sa = oracle.quant_rows(_host_bits(i["A"][:64]))
        a = oracle.dequant_rows(qa, sa)
        qb, sb = oracle.quant_rows(_host_bits(self.expert0_gate_up()))
        b = oracle.dequant_rows(qb, sb)
        rows, t_g = 0, 0.0
        while t_g < budget_s and rows < a.shape[0]:
            t0 = time.perf_counter()
            oracle.gemm(a, b, rows=np.array([rows], dtype=np.int64))
            t_g += time.perf_counter() - t0
            rows += 1
        tg = t_g / (2.0 * rows * 2 * self.I * self.H)
        elems = self.Mt * (self.H + self.I) + self.G * 2 * self.I * self.H + self.G * self.H * self.I
        return tq * elems + tg * self.gemm_flops, (
            f"oracle row quant of 256 routed rows and FP64 GEMM of {rows} rows against one expert "
            f"(N {2 * self.I}, K {self.H}); extrapolated to the full step")


class MoETrain(Workload):
    """One MoE expert-layer training pass over the 128-expert workload:
    forward (gate_up, down), dgrad (dA = dY1 W_gu, dH = dY2 W_dn) and wgrad
    (dW_gu = dY1^T A, dW_dn = dY2^T H) per expert.  dY1 / dY2 are synthetic
    output gradients (the activation between the projections is not part of
    the MXFP8 path)."""
    state_keys = ("W_gate_up", "W_down")

    def __init__(self, dev=None, tokens=16384, experts=128, name="moe_train"):
        import torch
        from mxfp8_microscaled_precision_gb300 import mxq, workloads
        self.name = name
        d = workloads.moe_grouped(dev or "cpu", tokens=tokens, experts=experts, weights=False)
        G, H, I = experts, 4096, 2048
        self.G, self.H, self.I = G, H, I
        self.Mt = d["A"].shape[0]
        w = "moe_grouped"
        seed_gu, seed_dn = workloads.seed_for(w, "W"), workloads.seed_for(w, "W_down")
        if dev is None:
            self.inputs = {"A": d["A"], "Hd": d["H"],
                           "W_gate_up": workloads.normal((2 * I, H), 0.02, seed_gu)}
            return
        Mt = self.Mt
        self.offsets = d["routing"].offsets.to(dev)
        self.inputs = {"A": d["A"], "Hd": d["H"], "offsets": self.offsets,
                       "W_gate_up": workloads.normal((G, 2 * I, H), 0.02, seed_gu, device=dev),
                       "W_down": workloads.normal((G, H, I), 0.02, seed_dn, device=dev),
                       "dY1": workloads.normal((Mt, 2 * I), 1e-3, seed_gu + 50, device=dev),
                       "dY2": workloads.normal((Mt, H), 1e-3, seed_dn + 50, device=dev)}
        u8 = dict(dtype=torch.uint8, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        sb = mxq.scale_bytes
        self.cap = mxq.grouped_capacity(Mt, G)
        cap = self.cap

        def rows(r, c):
            return (torch.empty((r, c), **u8), torch.empty(sb(r, c), **u8), None, None)

        def cols_g(c):
            return torch.empty((c, cap), **u8), torch.empty(sb(c, cap), **u8)
        self.qa, self.qh = rows(Mt, H), rows(Mt, I)
        self.qg1, self.qg2 = rows(Mt, 2 * I), rows(Mt, H)
        self.wgu = (torch.empty((G, 2 * I, H), **u8), torch.empty((G, sb(2 * I, H)), **u8),
                    torch.empty((G, H, 2 * I), **u8), torch.empty((G, sb(H, 2 * I)), **u8))
        self.wdn = (torch.empty((G, H, I), **u8), torch.empty((G, sb(H, I)), **u8),
                    torch.empty((G, I, H), **u8), torch.empty((G, sb(I, H)), **u8))
        self.c_g1, self.c_a, self.c_g2, self.c_h = cols_g(2 * I), cols_g(H), cols_g(H), cols_g(I)
        self.sa_g, self.sh_g, self.sg1_g, self.sg2_g = _group_tiled_setup(self, d["routing"].offsets,
                                                                          (H, I, 2 * I, H), dev)
        self.y1, self.y2 = torch.empty((Mt, 2 * I), **bf), torch.empty((Mt, H), **bf)
        self.da, self.dh = torch.empty((Mt, H), **bf), torch.empty((Mt, I), **bf)
        self.dwgu, self.dwdn = torch.empty((G, 2 * I, H), **bf), torch.empty((G, H, I), **bf)
        self.outputs = [self.y1, self.y2, self.da, self.dh, self.dwgu, self.dwdn]

    @property
    def gemm_flops(self):
        return 3 * (2 * self.Mt * 2 * self.I * self.H + 2 * self.Mt * self.H * self.I)

    def _quant_batched(self, w, out):
        from mxfp8_microscaled_precision_gb300 import mxq
        B, R, C = w.shape
        lib = mxq.lib()
        mxq._check(lib.mxq_quant_1x32_dual_batched(mxq._ptr(w), B, R, C, w.stride(1), w.stride(0),
                                                   *[mxq._ptr(t) for t in out], 1, 0, mxq._stream()),
                   "mxq_quant_1x32_dual_batched")

    def _quant_cols(self, x, out):
        from mxfp8_microscaled_precision_gb300 import mxq
        lib = mxq.lib()
        R, C = x.shape
        mxq._check(lib.mxq_quant_1x32_cols_grouped(mxq._ptr(x), R, C, x.stride(0), mxq._ptr(self.offsets),
                                                   self.G, self.cap, mxq._ptr(out[0]), mxq._ptr(out[1]), 1,
                                                   mxq._stream()), "mxq_quant_1x32_cols_grouped")

    def kernels(self):
        from mxfp8_microscaled_precision_gb300 import mxq
        i, G, H, I, Mt, off = self.inputs, self.G, self.H, self.I, self.Mt, self.offsets
        wgu, wdn = self.wgu, self.wdn
        f_gu, f_dn = 2 * Mt * 2 * I * H, 2 * Mt * H * I

        def colsb(c):
            return Mt * c * 3 + Mt * c // 32
        return [
            ("quant_A_row", "quant", _row_bytes(Mt, H), lambda: mxq.quant_1x32_dual(i["A"], col=False, out=self.qa)),
            ("quant_H_row", "quant", _row_bytes(Mt, I), lambda: mxq.quant_1x32_dual(i["Hd"], col=False, out=self.qh)),
            ("regroup_A_scales", "layout", _regroup_bytes(self, H),
             lambda: mxq.scale_regroup_rows(self.qa[1], Mt, H, off, self.gt_cap, out=self.sa_g)),
            ("regroup_H_scales", "layout", _regroup_bytes(self, I),
             lambda: mxq.scale_regroup_rows(self.qh[1], Mt, I, off, self.gt_cap, out=self.sh_g)),
            ("quant_Wgu_dual", "quant", _dual_bytes(G * 2 * I, H), lambda: self._quant_batched(i["W_gate_up"], wgu)),
            ("quant_Wdn_dual", "quant", _dual_bytes(G * H, I), lambda: self._quant_batched(i["W_down"], wdn)),
            ("grouped_fwd_gate_up", "gemm", f_gu,
             lambda: mxq.grouped_gemm_group_tiled(self.qa[0], self.sa_g, wgu[0].view(G * 2 * I, H), wgu[1].view(-1),
                                                  off, 2 * I, H, self.gt_cap, out=self.y1)),
            ("grouped_fwd_down", "gemm", f_dn,
             lambda: mxq.grouped_gemm_group_tiled(self.qh[0], self.sh_g, wdn[0].view(G * H, I), wdn[1].view(-1),
                                                  off, H, I, self.gt_cap, out=self.y2)),
            ("quant_dY1_row", "quant", _row_bytes(Mt, 2 * I), lambda: mxq.quant_1x32_dual(i["dY1"], col=False, out=self.qg1)),
            ("quant_dY2_row", "quant", _row_bytes(Mt, H), lambda: mxq.quant_1x32_dual(i["dY2"], col=False, out=self.qg2)),
            ("regroup_dY1_scales", "layout", _regroup_bytes(self, 2 * I),
             lambda: mxq.scale_regroup_rows(self.qg1[1], Mt, 2 * I, off, self.gt_cap, out=self.sg1_g)),
            ("regroup_dY2_scales", "layout", _regroup_bytes(self, H),
             lambda: mxq.scale_regroup_rows(self.qg2[1], Mt, H, off, self.gt_cap, out=self.sg2_g)),
            ("grouped_dgrad_gate_up", "gemm", f_gu,
             lambda: mxq.grouped_gemm_group_tiled(self.qg1[0], self.sg1_g, wgu[2].view(G * H, 2 * I), wgu[3].view(-1),
                                                  off, H, 2 * I, self.gt_cap, out=self.da)),
            ("grouped_dgrad_down", "gemm", f_dn,
             lambda: mxq.grouped_gemm_group_tiled(self.qg2[0], self.sg2_g, wdn[2].view(G * I, H), wdn[3].view(-1),
                                                  off, I, H, self.gt_cap, out=self.dh)),
            ("quant_dY1_cols", "quant", colsb(2 * I), lambda: self._quant_cols(i["dY1"], self.c_g1)),
            ("quant_A_cols", "quant", colsb(H), lambda: self._quant_cols(i["A"], self.c_a)),
            ("quant_dY2_cols", "quant", colsb(H), lambda: self._quant_cols(i["dY2"], self.c_g2)),
            ("quant_H_cols", "quant", colsb(I), lambda: self._quant_cols(i["Hd"], self.c_h)),
            ("grouped_wgrad_gate_up", "gemm", f_gu,
             lambda: mxq.grouped_gemm_wgrad(self.c_g1[0], self.c_g1[1], self.c_a[0], self.c_a[1], off, Mt, out=self.dwgu)),
            ("grouped_wgrad_down", "gemm", f_dn,
             lambda: mxq.grouped_gemm_wgrad(self.c_g2[0], self.c_g2[1], self.c_h[0], self.c_h[1], off, Mt, out=self.dwdn)),
        ]

    def expert0_gate_up(self):
        w = self.inputs["W_gate_up"]
        return w[0] if w.dim() == 3 else w

    def cpu_sample(self, budget_s):
        # MoE.cpu_sample measures per-element and per-FLOP oracle rates and scales
        # the FLOP part by self.gemm_flops (here the whole training step).
        t_step, desc = MoE.cpu_sample(self, budget_s)
        return t_step, desc + " (GEMM rate applied to the forward + dgrad + wgrad FLOPs)"


def _host_bits(t):
    import numpy as np
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def make_workload(name, dev=None):
    """The workload on device `dev`, or host-only inputs when dev is None."""
    from mxfp8_microscaled_precision_gb300 import workloads
    if name == "linear_train":
        return LinearTrain(name, 8192, 4096, 4096, lambda d: workloads.linear_train(d), dev)
    if name.startswith("sweep_"):
        K = int(name.split("_")[1])
        return LinearTrain(name, 16384, K, K, lambda d: workloads.sweep(K, d), dev)
    if name == "linear_fwd_small":
        return LinearFwdSmall(dev)
    if name == "weight_32x32":
        return Weight32(dev)
    if name in ("linear_fwd_chain_fused", "linear_fwd_chain_two_pass"):
        return LinearFwdChain(name.endswith("fused"), dev)
    if name == "moe_grouped":
        return MoE(dev)
    if name == "moe_train":
        return MoETrain(dev)
    if name == "moe_train_small":   # 2048 tokens over 16 experts: the per-expert sizes of moe_train, a few GB
        return MoETrain(dev, tokens=2048, experts=16, name=name)
    if name in ("fsdp_mxfp8", "fsdp_mxfp8_32x32"):
        return FsdpWeight("mxfp8" if name == "fsdp_mxfp8" else "mxfp8-32x32", dev)
    raise SystemExit(f"unknown workload {name}")


WORKLOAD_NAMES = ["linear_train", "linear_fwd_small", "weight_32x32", "moe_grouped", "moe_train", "moe_train_small",
                  "fsdp_mxfp8", "fsdp_mxfp8_32x32", "linear_fwd_chain_fused", "linear_fwd_chain_two_pass",
                  "sweep_4096", "sweep_7168", "sweep_16384"]


def workload_config(w):
    cfg = {"workload": w.name}
    for k in ("M", "N", "K", "n", "k", "G", "H", "I", "Mt", "cap", "world", "recipe"):
        if hasattr(w, k):
            cfg[k] = getattr(w, k)
    cfg["l2"] = "flushed between timed steps (256 MB device write, outside the timed intervals)"
    return cfg


def cpu_model():
    """The host CPU's model name (from /proc/cpuinfo, else the machine type)."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "Hardware"):
            for line in info.splitlines():
                if line.split(":")[0].strip() == key and ":" in line:
                    return line.split(":", 1)[1].strip()
        parts = sorted({line.split(":", 1)[1].strip() for line in info.splitlines()
                        if line.startswith("CPU part") and ":" in line})
        if parts:
            return f"{platform.machine()} (CPU part {', '.join(parts)})"
    except OSError:
        pass
    return platform.machine() or "unknown"


def vendor_mxfp8_tflops(dev, shapes):
    """The vendor library's MXFP8 GEMM (PyTorch _scaled_mm with float8_e4m3fn
    operands and E8M0 block scales, cuBLASLt underneath) timed at each shape:
    {"MxNxK": TFLOP/s}, or {"error": why}.  A denominator only: none of the
    hot path runs here, and its outputs are not used."""
    import torch
    if not hasattr(torch, "float8_e8m0fnu"):
        return {"error": "this PyTorch has no float8_e8m0fnu"}
    out = {}
    for (M, N, K) in shapes:
        try:
            a = torch.randint(-100, 100, (M, K), device=dev, dtype=torch.int8).view(torch.uint8)
            a = (a & 0x77).view(torch.float8_e4m3fn)       # finite codes only
            b = (torch.randint(0, 255, (N, K), device=dev, dtype=torch.uint8) & 0x77).view(torch.float8_e4m3fn)
            sa = torch.full(((M + 127) // 128 * 128, (K // 32 + 3) // 4 * 4), 127, dtype=torch.uint8,
                            device=dev).view(torch.float8_e8m0fnu)
            sb = torch.full(((N + 127) // 128 * 128, (K // 32 + 3) // 4 * 4), 127, dtype=torch.uint8,
                            device=dev).view(torch.float8_e8m0fnu)
            f = lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
            for _ in range(3):
                f()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(5, min(50, int(2e12 / (2.0 * M * N * K)) + 1))
            e0.record()
            for _ in range(reps):
                f()
            e1.record()
            torch.cuda.synchronize()
            out[f"{M}x{N}x{K}"] = round(2.0 * M * N * K * reps / (e0.elapsed_time(e1) / 1e3) / 1e12, 1)
            del a, b, sa, sb
        except Exception as ex:                              # noqa: BLE001 -- a denominator, not the product
            out[f"{M}x{N}x{K}"] = None
            out.setdefault("error", f"{type(ex).__name__}: {str(ex).splitlines()[0][:160]}")
    torch.cuda.empty_cache()
    return out


def vendor_mxfp8_sustained(dev, shape, seconds, operands):
    """The vendor library's MXFP8 GEMM at one shape on the workload's own
    quantized operands (payload bytes and MMA-tiled scale bytes of A [M, K] and
    B [N, K], so that its power draw follows the same data), launched back to
    back for about `seconds` (the length of this run's timed region): the power
    state a long step reaches.  {"shape", "tflops", "seconds", "clocks"} or
    {"error": why}.  A comparison only, beside the burst peak."""
    import torch
    if not hasattr(torch, "float8_e8m0fnu"):
        return {"error": "this PyTorch has no float8_e8m0fnu"}
    M, N, K = shape
    try:
        a_q, a_s, b_q, b_s = operands
        a, b = a_q.view(torch.float8_e4m3fn), b_q.view(torch.float8_e4m3fn)
        sa = a_s.view(torch.float8_e8m0fnu).view((M + 127) // 128 * 128, -1)
        sb = b_s.view(torch.float8_e8m0fnu).view((N + 127) // 128 * 128, -1)
        f = lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        f()
        e1.record()
        torch.cuda.synchronize()
        reps = max(10, int(seconds / max(e0.elapsed_time(e1) / 1e3, 1e-6)))
        sampler = ClockSampler(dev.index)
        sampler.start()
        time.sleep(0.2)
        t_w0 = time.time()
        e0.record()
        for _ in range(reps):
            f()
        e1.record()
        torch.cuda.synchronize()
        t_w1 = time.time()
        sampler.stop()
        ms = e0.elapsed_time(e1)
        return {"shape": f"{M}x{N}x{K}", "operands": "the workload's quantized X and W", "tflops": round(2.0 * M * N * K * reps / (ms / 1e3) / 1e12, 1),
                "seconds": round(ms / 1e3, 3), "launches": reps, "clocks": sampler.summary(t_w0 - 0.05, t_w1 + 0.05)}
    except Exception as ex:                              # noqa: BLE001 -- a comparison, not the product
        return {"error": f"{type(ex).__name__}: {str(ex).splitlines()[0][:160]}"}


# ---- the GPU arm ---------------------------------------------------------------------------

def time_device(w, args, dev, world):
    """Warm-up, then args.steps timed steps of workload w with the inputs
    resident in HBM (CUDA events per step and per kernel on the launching
    stream, L2 flushed between steps) while nvidia-smi samples the clocks.
    Returns the per-kernel and per-step times and the clock summary."""
    import torch
    from mxfp8_microscaled_precision_gb300 import mxq
    kern = w.kernels()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.fill_(1)
        for (_, _, _, fn) in kern:
            fn()
    torch.cuda.synchronize()
    st = mxq.get_device_status()
    if st != 0:
        raise SystemExit(f"device status {st} after warm-up of {w.name}")
    nk = len(kern)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    barrier(dev)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for s in range(args.steps):
        flush.fill_(s & 0xFF)                      # evict L2 between steps (not timed)
        ev[s][0].record(stream)
        for j, (_, _, _, fn) in enumerate(kern):
            fn()
            ev[s][j + 1].record(stream)
    torch.cuda.synchronize()
    barrier(dev)
    t_wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    st = mxq.get_device_status()
    if st != 0:
        raise SystemExit(f"device status {st} after the timed steps of {w.name}")
    per_kernel = [[ev[s][j].elapsed_time(ev[s][j + 1]) for s in range(args.steps)] for j in range(nk)]
    step_ms = [ev[s][0].elapsed_time(ev[s][nk]) for s in range(args.steps)]
    return {"kern": kern, "per_kernel": per_kernel, "step_ms": step_ms, "flush": flush,
            "clocks": sampler.summary(t_wall0 - 0.05, t_wall1 + 0.05)}


def rates(t, steps, peaks, gemm_peak):
    """GEMM and quantizer rates of one timed workload against their peaks."""
    kern, per_kernel = t["kern"], t["per_kernel"]
    nk = len(kern)
    gemm_idx = [j for j in range(nk) if kern[j][1] == "gemm"]
    quant_idx = [j for j in range(nk) if kern[j][1] == "quant"]
    gemm_s = sum(sum(per_kernel[j]) for j in gemm_idx) / 1e3
    quant_s = sum(sum(per_kernel[j]) for j in quant_idx) / 1e3
    gemm_tflops = sum(kern[j][2] for j in gemm_idx) * steps / gemm_s / 1e12
    quant_gbs = sum(kern[j][2] for j in quant_idx) * steps / quant_s / 1e9 if quant_idx else 0.0
    other_hbm = {}
    for j in range(nk):
        if kern[j][1] not in ("gemm", "quant"):
            gbs = kern[j][2] * steps / (sum(per_kernel[j]) / 1e3) / 1e9
            other_hbm[kern[j][0]] = {"kind": kern[j][1], "bytes_per_launch": kern[j][2],
                                     "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    return {"gemm_tflops": gemm_tflops, "gemm_frac": gemm_tflops / gemm_peak, "quant_gbs": quant_gbs,
            "quant_frac": quant_gbs / peaks["hbm_gbs"],
            "per_launch_flops": statistics.mean(kern[j][2] for j in gemm_idx),
            "kernels_ms": {kern[j][0]: round(statistics.mean(per_kernel[j]), 5) for j in range(nk)},
            "kernels_ms_median": {kern[j][0]: round(statistics.median(per_kernel[j]), 5) for j in range(nk)},
            "other_hbm": other_hbm}


def gemm_peak_of(peaks, vendor):
    """The GEMM denominator: the larger of 2 x the measured BF16 burst (the
    nominal FP8/BF16 ratio) and the best vendor MXFP8 rate timed in this run."""
    fp8_nominal = peaks["bf16_tflops"] * FP8_OVER_BF16
    best = max([v for k, v in vendor.items() if k != "error" and v], default=0.0)
    if best > fp8_nominal:
        return best, f"vendor MXFP8 GEMM (cuBLASLt via torch._scaled_mm) timed in this run, best of {vendor}"
    return fp8_nominal, (f"{peaks['source']} bf16 burst x {FP8_OVER_BF16:g} (nominal fp8/bf16 ratio); "
                         f"vendor MXFP8 in this run {vendor}")


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from mxfp8_microscaled_precision_gb300 import build as mbuild, mxq
    mbuild.build()
    mxq.lib()
    peaks = load_peaks()
    w = make_workload(args.workload, dev)
    vendor_shapes = list(VENDOR_SHAPES)
    if all(hasattr(w, k) for k in ("M", "N", "K")) and (w.M, w.N, w.K) not in vendor_shapes:
        vendor_shapes.append((w.M, w.N, w.K))
    vendor = vendor_mxfp8_tflops(dev, vendor_shapes) if not args.no_vendor_peak else {"error": "not timed"}
    gemm_peak, gemm_peak_source = gemm_peak_of(peaks, vendor)
    fp8_nominal = peaks["bf16_tflops"] * FP8_OVER_BF16

    t = time_device(w, args, dev, world)
    kern, stream, flush = t["kern"], torch.cuda.current_stream(), t["flush"]
    main_clocks = t["clocks"]
    nk = len(kern)
    total_s = sum(t["step_ms"]) / 1e3
    step_median_ms = statistics.median(t["step_ms"])
    max_total_s = max_over_ranks(total_s, dev if world > 1 else None)
    value = aggregate_value(w.gemm_flops, args.steps, world, max_total_s)
    r = rates(t, args.steps, peaks, gemm_peak)
    roofline = {"bound": "tensor", "kernel": "gemm_mxf8_pair_kernel", "achieved": round(r["gemm_tflops"], 1),
                "peak": round(gemm_peak, 1), "unit": "TFLOP/s", "frac": round(r["gemm_frac"], 4),
                "traffic": GEMM_TRAFFIC_BYTES.get(w.name),
                "units_per_launch": r["per_launch_flops"],
                "peak_source": gemm_peak_source,
                "frac_of_2x_bf16_burst": round(r["gemm_tflops"] / fp8_nominal, 4)}
    roofline_quant = {"bound": "hbm", "kernel": "quant kernels", "achieved": round(r["quant_gbs"], 1),
                      "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(r["quant_frac"], 4),
                      "peak_source": peaks["source"] + " copy bandwidth"}
    own_launches = sum(LAUNCHES_PER_ENTRY.get(kern[j][0], 1) for j in range(nk) if kern[j][1] != "collective")

    # ---- end to end through the public API, host buffers, copies inside the timed step
    # Every step copies its inputs from pinned host memory and its outputs back. Steps
    # are pipelined the way a training loop would run them: two device copies of the
    # workload alternate, so the host-to-device copy of step s+1 and the device-to-host
    # copy of step s-1 overlap the kernels of step s (three streams, event-ordered).
    e2e = None
    if not args.no_e2e:
        host_in = {k: v.detach().cpu().pin_memory() for k, v in w.inputs.items() if k not in w.state_keys}
        host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in w.outputs]
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(o.numel() * o.element_size() for o in host_out)
        flush_each = h2d <= L2_BYTES                    # inputs not larger than L2: flush between steps
        inst = [(w, kern), None]
        w2 = make_workload(args.workload, dev)
        inst[1] = (w2, w2.kernels())
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        n_e2e = args.steps

        def run_pipeline(n, t_events=None):
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_cmp = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            if t_events:
                t_events[0].record(s_in)
            for i in range(n):
                wi, ki = inst[i % 2]
                if i >= 2:
                    s_in.wait_event(ev_cmp[i - 2])          # the inputs of this copy were consumed
                with torch.cuda.stream(s_in):
                    for k, v in host_in.items():
                        wi.inputs[k].copy_(v, non_blocking=True)
                ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                if i >= 2:
                    stream.wait_event(ev_out[i - 2])        # the outputs of this copy were read back
                if flush_each:
                    flush.fill_(i & 0xFF)
                for (_, _, _, fn) in ki:
                    fn()
                ev_cmp[i].record(stream)
                s_out.wait_event(ev_cmp[i])
                with torch.cuda.stream(s_out):
                    for o, h in zip(wi.outputs, host_out):
                        h.copy_(o, non_blocking=True)
                ev_out[i].record(s_out)
            if t_events:
                t_events[1].record(s_out)
            torch.cuda.synchronize()

        run_pipeline(4)                                     # warm-up of both copies
        tev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        barrier(dev)
        run_pipeline(n_e2e, tev)
        e2e_total = tev[0].elapsed_time(tev[1]) / 1e3
        e2e_total = max_over_ranks(e2e_total, dev if world > 1 else None)
        e2e = {"value": round(aggregate_value(w.gemm_flops, n_e2e, world, e2e_total), 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_total / n_e2e * 1e3, 4),
               "pipelining": "2 alternating device copies; copies of neighbouring steps overlap the kernels",
               "resident": list(w.state_keys),
               "l2": "flushed before each step's kernels" if flush_each else
                     "each step's inputs (larger than L2) arrive fresh from the host"}
        del w2, inst, host_in, host_out
        st = mxq.get_device_status()
        if st != 0:
            raise SystemExit(f"device status {st} after the end-to-end steps")

    # ---- the workload's quantizers timed alone (same kernels and sizes, no GEMM
    # between them): the in-step rate above follows the GEMMs' power draw, which
    # lowers the clock the quantizers then run at
    quant_alone = None
    quant_alone_launches = 0
    quant_kern = [k for k in kern if k[1] == "quant"]
    if quant_kern and not args.no_quant_alone:
        # the power state the GEMMs leave takes tens of milliseconds to settle: idle first
        torch.cuda.synchronize()
        time.sleep(1.0)
        ev_q = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for s in range(args.warmup):
            flush.fill_(s & 0xFF)
            for (_, _, _, fn) in quant_kern:
                fn()
        torch.cuda.synchronize()
        sampler_q = ClockSampler(dev.index)
        sampler_q.start()
        time.sleep(0.3)
        tq0 = time.time()
        for s in range(args.steps):
            flush.fill_(s & 0xFF)
            ev_q[s][0].record(stream)
            for (_, _, _, fn) in quant_kern:
                fn()
            ev_q[s][1].record(stream)
        torch.cuda.synchronize()
        tq1 = time.time()
        time.sleep(0.2)
        sampler_q.stop()
        q_s = sum(e[0].elapsed_time(e[1]) for e in ev_q) / 1e3
        q_gbs = sum(k[2] for k in quant_kern) * args.steps / q_s / 1e9
        quant_alone = {"bound": "hbm", "kernel": "quant kernels (timed alone)", "achieved": round(q_gbs, 1),
                       "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(q_gbs / peaks["hbm_gbs"], 4),
                       "peak_source": peaks["source"] + " copy bandwidth",
                       "clocks": sampler_q.summary(tq0 - 0.05, tq1 + 0.05),
                       "how": "the step's quantizer launches only, after 1 s idle, L2 flushed before each step, "
                              "CUDA events"}
        quant_alone_launches = args.steps * sum(LAUNCHES_PER_ENTRY.get(k[0], 1) for k in quant_kern)

    # ---- the vendor's MXFP8 GEMM at this workload's shape, back to back for as
    # long as the timed region above: the same power state as a long step
    vendor_sustained = None
    if not args.no_vendor_peak and all(hasattr(w, k) for k in ("M", "N", "K", "qx", "qw")):
        torch.cuda.synchronize()
        time.sleep(1.0)
        vendor_sustained = vendor_mxfp8_sustained(dev, (w.M, w.N, w.K), max(0.2, total_s),
                                                  (w.qx[0], w.qx[1], w.qw[0], w.qw[1]))
        if "tflops" in vendor_sustained:
            roofline["frac_of_vendor_sustained"] = round(r["gemm_tflops"] / vendor_sustained["tflops"], 4)

    # ---- further workloads timed in the same process (device side only)
    extra = {}
    extra_launches = 0
    del t, flush
    for name in [n for n in args.extra_workloads.split(",") if n and n != "none" and n != args.workload]:
        torch.cuda.empty_cache()
        wx = make_workload(name, dev)
        tx = time_device(wx, args, dev, world)
        rx = rates(tx, args.steps, peaks, gemm_peak)
        tot_x = max_over_ranks(sum(tx["step_ms"]) / 1e3, dev if world > 1 else None)
        extra[name] = {"config": workload_config(wx),
                       "value": round(aggregate_value(wx.gemm_flops, args.steps, world, tot_x), 2),
                       "unit": "TFLOP/s", "ms_per_step": round(tot_x / args.steps * 1e3, 4),
                       "gemm_tflops": round(rx["gemm_tflops"], 1), "gemm_frac_peak": round(rx["gemm_frac"], 4),
                       "gemm_frac_of_2x_bf16_burst": round(rx["gemm_tflops"] / fp8_nominal, 4),
                       "quant_tbs": round(rx["quant_gbs"] / 1e3, 3), "quant_frac_hbm": round(rx["quant_frac"], 4),
                       "kernels_ms": rx["kernels_ms"], "clocks": tx["clocks"]}
        if rx["other_hbm"]:
            extra[name]["hbm_kernels"] = rx["other_hbm"]
        extra_launches += args.steps * sum(LAUNCHES_PER_ENTRY.get(k[0], 1) for k in tx["kern"] if k[1] != "collective")
        del wx, tx

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_budget)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(max_total_s / args.steps * 1e3, 4),
                "ms_per_step_median": round(step_median_ms, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3 (E8M0 block scales, fp32 accumulate)",
                "data": "synthetic (seeded generators; shapes of the linear / MoE-expert workloads)",
                "config": workload_config(w),
                "gemm_tflops": round(r["gemm_tflops"], 1), "gemm_frac_peak": round(r["gemm_frac"], 4),
                "quant_tbs": round(r["quant_gbs"] / 1e3, 3), "quant_frac_hbm": round(r["quant_frac"], 4),
                "kernels_ms": r["kernels_ms"], "kernels_ms_median": r["kernels_ms_median"],
                "roofline": roofline, "roofline_quant": roofline_quant, "roofline_quant_alone": quant_alone,
                "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": own_launches * args.steps + extra_launches + quant_alone_launches,
                "gpu_launches_split": {w.name: own_launches * args.steps, "extra_workloads": extra_launches,
                                       "quant_alone": quant_alone_launches},
                "clocks": main_clocks, "vendor_mxfp8_tflops": vendor,
                "vendor_mxfp8_sustained": vendor_sustained, "impl": "mxq"}
        if r["other_hbm"]:
            line["hbm_kernels"] = r["other_hbm"]
        if hasattr(w, "extra"):
            line.update(w.extra())
        for name, block in extra.items():
            line["moe_block" if name == "moe_grouped" else "extra_" + name] = block
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def cpu_baseline(w, budget_s):
    from oracle import oracle
    oracle.build()
    t_step, sample = w.cpu_sample(budget_s)
    cores = _omp_threads()
    return {"value": round(w.gemm_flops / t_step / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "cpu_model": cpu_model(), "kind": "oracle", "sample": sample,
            "extrapolated_s_per_step": round(t_step, 3)}


def _omp_threads():
    v = os.environ.get("OMP_NUM_THREADS")
    if v and v.isdigit():
        return int(v)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---- the reference arm: the oracle on the host cores ------------------------------------------

def run_reference(args):
    """The oracle timed on the host cores.  Each step is one bounded sample of
    the workload (cpu_sample); `ms_per_step` is the measured wall time of those
    samples, `value` the rate they give for the full step (sampled rates
    extrapolated to the step's work), and `extrapolated_ms_per_full_step` the
    time a whole step would take at those rates."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import oracle
    oracle.build()
    w = make_workload(args.workload)
    per_step_budget = max(0.05, min(4.0, 100.0 / max(1, args.steps + args.warmup)))
    ext, wall = [], []
    desc = ""
    t_run0 = time.perf_counter()
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        t, desc = w.cpu_sample(per_step_budget * 0.8)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            ext.append(t)
            wall.append(dt)
    t_full = statistics.mean(ext)
    value = w.gemm_flops / t_full / 1e12
    cores = _omp_threads()
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(wall) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "config": workload_config(w), "impl": "reference",
            "extrapolated_ms_per_full_step": round(t_full * 1e3, 3),
            "wall_s_all_steps": round(time.perf_counter() - t_run0, 3),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
                             "kind": "oracle",
                             "sample": desc + "; each timed step is this bounded sample (ms_per_step is its "
                                              "measured wall time; value is the sample's rate over the full "
                                              "step's work)"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile_gemm(shape):
    """One launch of this library's dense MXFP8 GEMM and one of the vendor's
    (torch._scaled_mm, E4M3 operands, E8M0 scales) at M x N x K on the same
    random operands, for a profiler to capture side by side; prints the largest
    difference of the two BF16 outputs."""
    import torch
    from mxfp8_microscaled_precision_gb300 import build as mbuild, mxq
    mbuild.build()
    M, N, K = (int(v) for v in shape.split("x"))
    dev = torch.device("cuda:0")
    a = torch.randint(0, 256, (M, K), device=dev, dtype=torch.uint8) & 0x77      # finite E4M3 codes
    b = torch.randint(0, 256, (N, K), device=dev, dtype=torch.uint8) & 0x77
    sa = torch.full((mxq.scale_bytes(M, K),), 120, dtype=torch.uint8, device=dev)
    sb = torch.full((mxq.scale_bytes(N, K),), 120, dtype=torch.uint8, device=dev)
    y = mxq.gemm(a, sa, b, sb, M, N, K)
    torch.cuda.synchronize()
    y2 = torch._scaled_mm(a.view(torch.float8_e4m3fn), b.view(torch.float8_e4m3fn).t(),
                          sa.view(torch.float8_e8m0fnu).view((M + 127) // 128 * 128, -1),
                          sb.view(torch.float8_e8m0fnu).view((N + 127) // 128 * 128, -1), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    print(json.dumps({"profile_gemm": shape, "max_abs_diff_vs_vendor": float((y.float() - y2.float()).abs().max())}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mxq", "reference"], default="mxq")
    ap.add_argument("--workload", choices=WORKLOAD_NAMES, default=DEFAULT_WORKLOAD)
    ap.add_argument("--extra-workloads", default=DEFAULT_EXTRA,
                    help="comma-separated workloads timed after the main one in the same process "
                         "(device side only), or 'none'")
    ap.add_argument("--no-quant-alone", action="store_true",
                    help="do not time the workload's quantizers alone (without the GEMMs between them)")
    ap.add_argument("--no-vendor-peak", action="store_true",
                    help="do not time the vendor MXFP8 GEMM (the GEMM peak is then 2 x the BF16 burst)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle GEMM in the CPU baseline")
    ap.add_argument("--profile-gemm", metavar="MxNxK",
                    help="launch this library's GEMM and the vendor's once each at this shape (for ncu) and exit")
    args = ap.parse_args(argv)
    if args.profile_gemm:
        return run_profile_gemm(args.profile_gemm)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
