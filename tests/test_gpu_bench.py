"""bench.py on the GPU, end to end, on the 128³ workload (50 FGP steps per
bench step): the JSON line carries every key of the contract with values
that follow from the workload (e2e bytes, launch counts, the roofline's
algorithmic bytes), and the reference arm describes the same workload with
the same config."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    out = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_bench_line_on_the_128_workload():
    import bench
    from fgp_dual_stencil_gb300 import synth
    w = synth.WORKLOADS["c2"]
    K, W = 3, 3
    d = run_bench("--workload", "c2", "--steps", str(K), "--warmup", str(W))
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "e2e", "clocks",
                "cpu_baseline"):
        assert key in d, key
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["n_gpus"] == 1 and d["steps"] == K and d["warmup"] == W
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["config"] == bench.workload_config(w, 1)
    assert d["value"] > 0 and abs(d["value"] - w.nvox * w.steps / (d["ms_per_step"] * 1e6)) < 0.01 * d["value"]
    # two-step launches for the 50 steps, and the primal, per bench step
    assert d["gpu_launches"] == K * (w.steps // 2 + 1)
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert rf["algorithmic_bytes_per_launch"] == 52 * w.nvox * 2
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] == 4 * w.nvox and e2e["d2h_bytes_per_step"] == 4 * w.nvox
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0
    if d["clocks"] is not None:
        assert d["clocks"]["samples"] >= 1 and d["clocks"]["sm_mhz"] > 0


def test_reference_arm_on_the_same_workload():
    import bench
    from fgp_dual_stencil_gb300 import synth
    d = run_bench("--impl", "reference", "--workload", "c2", "--steps", "1", "--warmup", "0")
    assert d["impl"] == "reference" and d["gpu_launches"] == 0
    assert d["config"] == bench.workload_config(synth.WORKLOADS["c2"], 1)
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
