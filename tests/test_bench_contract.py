"""The JSON line bench.py prints for the reference arm (the CPU oracle), on CPU:
one line with the metric, unit, config and the baseline fields the contract
names, values consistent with each other."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "linear_fwd_small",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "linear_fwd_small"
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert cb["cpu_model"]
    # ms_per_step is the measured time of what ran: the timed steps fit in the run's own wall time
    assert d["steps"] * d["ms_per_step"] <= d["wall_s_all_steps"] * 1e3 * 1.01
    assert d["extrapolated_ms_per_full_step"] > 0
    e = d["e2e"]
    assert e["value"] == d["value"] and e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_default_workload_is_the_largest_single_gpu_config():
    import bench
    ap_default = bench.DEFAULT_WORKLOAD
    assert ap_default == "sweep_16384" and bench.DEFAULT_EXTRA == "moe_grouped"


def test_gemm_peak_is_not_below_the_vendor_rate():
    import bench
    peaks = {"bf16_tflops": 1900.0, "source": "measured"}
    p, src = bench.gemm_peak_of(peaks, {"8192x4096x4096": 3650.0, "16384x8192x8192": 4190.0})
    assert p == 4190.0 and "vendor" in src
    p, src = bench.gemm_peak_of(peaks, {"error": "no e8m0"})
    assert p == 3800.0 and "bf16" in src


def test_rejects_too_few_warmup_steps():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_group_tiled_band_accounting():
    """The bench's regroup bytes and buffers use the bands the oracle's group-tiled
    layout fills (each expert ceil(n_g / 128) bands) and the capacity the C ABI
    asks for (ceil(rows / 128) + G bands)."""
    import numpy as np
    import bench
    from oracle import oracle

    class W:
        pass
    w = W()
    w.Mt, w.G = 1000, 4
    off = [0, 130, 130, 700, 1000]
    bufs = bench._group_tiled_setup(w, off, (256, 128), "cpu")
    filled = oracle.scale_group_tiled(np.zeros((1000, 8), np.uint8), off).size
    assert w.gt_bands * 2 * 512 == filled
    assert w.gt_cap == (1000 + 127) // 128 + 4
    assert bufs[0].numel() == w.gt_cap * 2 * 512 and bufs[1].numel() == w.gt_cap * 512
    assert bench._regroup_bytes(w, 256) == ((1000 + 127) // 128 + w.gt_bands) * 2 * 512
