"""Host logic of bench.py that decides what the JSON line reports: the kernel
source hash that gates the recorded DRAM traffic (comment edits keep it,
code edits drop the traffic to null) and the scaling of that traffic to a
volume; the workload description both arms share."""
import json
import os
import shutil

import bench


def test_strip_comments_keeps_code_and_strings():
    src = 'int a; // tail\n/* block\n spanning */ int b = 1; /**/\n\n  const char *s = "// not a comment";\n'
    out = bench._strip_comments(src)
    assert out == 'int a;\n int b = 1;\n  const char *s = "// not a comment";'
    assert bench._strip_comments('char q = "a\\"//b"; // c') == 'char q = "a\\"//b";'


def _tree(tmp_path):
    """A copy of the hashed sources and of the recorded traffic in tmp_path."""
    src = os.path.join(bench.ROOT, "fgp_dual_stencil_gb300", "csrc")
    dst = tmp_path / "fgp_dual_stencil_gb300" / "csrc"
    dst.mkdir(parents=True)
    for fn in ("fgp_kernels.cuh", "zmarch_tma.cuh", "zmarch2_tma.cuh"):
        shutil.copy(os.path.join(src, fn), dst / fn)
    (tmp_path / "profiles").mkdir()
    return dst


def test_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    rec = {"fgp_step2_zmarch_tma": {"source_hash": h, "dram_bytes_per_voxel": 54.5}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("fgp_step2_zmarch_tma", 1000) == 54500.0
    assert bench.ncu_traffic("fgp_step_zmarch_tma", 1000) is None          # not recorded

    k = csrc / "zmarch2_tma.cuh"
    k.write_text(k.read_text() + "\n// a comment added at the end\n")
    assert bench.kernel_source_hash() == h                                  # comments: same
    assert bench.ncu_traffic("fgp_step2_zmarch_tma", 1000) == 54500.0

    k.write_text(k.read_text() + "\nstatic const int changed = 1;\n")
    assert bench.kernel_source_hash() != h                                  # code: new hash
    assert bench.ncu_traffic("fgp_step2_zmarch_tma", 1000) is None

    (tmp_path / "profiles" / "traffic.json").write_text("{not json")
    assert bench.ncu_traffic("fgp_step2_zmarch_tma", 1000) is None


def test_committed_traffic_names_the_bench_kernels():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for name in ("fgp_step2_zmarch_tma", "fgp_step_zmarch_tma", "fgp_step_zmarch_tma<__half>"):
        ent = rec[name]
        assert len(ent["source_hash"]) == 16 and ent["dram_bytes_per_voxel"] > 0
        assert "--clock-control none" in ent["command"]


def test_roofline_reports_the_model_and_the_measured_dram_fraction():
    # a two-step launch of 512^3 voxels: 104 B per voxel by the model, 52.8 B measured
    n = 512 ** 3
    r = bench.roofline_entry("fgp_step2_zmarch_tma", 104 * n, 1.25e-3, 6795.5, "measured", 52.8 * n, 2.0, 52)
    assert r["frac"] == r["model_frac"] == round(104 * n / 1.25e-3 / 1e9 / 6795.5, 4)
    assert r["frac"] > 1.0 and r["model_frac_basis"].startswith("2 FGP step(s) per launch, 52 B")
    assert r["dram_achieved"] == round(52.8 * n / 1.25e-3 / 1e9, 1)
    assert r["dram_frac"] == round(52.8 * n / 1.25e-3 / 1e9 / 6795.5, 4) and r["dram_frac"] < 1.0
    assert r["traffic"] == round(52.8 * n) and r["bound"] == "hbm" and r["unit"] == "GB/s"
    none = bench.roofline_entry("fgp_step2_zmarch_tma", 104 * n, 1.25e-3, 6800.0, "fallback", None, 2.0, 52)
    assert none["traffic"] is None and none["dram_frac"] is None and none["dram_achieved"] is None
    assert none["peak_source"] == "fallback 6.8 TB/s"


def test_reference_arm_reports_the_same_config_as_the_library_arm(monkeypatch):
    """The oracle's arm runs on the small workload here and must describe the
    workload with the very dictionary the library's arm puts in "config"."""
    import sys
    from fgp_dual_stencil_gb300 import synth
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--workload", "c1",
                                      "--steps", "1", "--warmup", "0"])
    line = bench.reference_arm(bench.parse_args(), 1, 0)
    assert line["impl"] == "reference" and line["gpu_launches"] == 0
    assert line["config"] == bench.workload_config(synth.WORKLOADS["c1"], 1)
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    for wl in synth.WORKLOADS.values():
        cfg = bench.workload_config(wl, 1)
        assert set(cfg) == {"workload", "nx", "ny", "nz", "fgp_steps_per_bench_step", "l2", "parallelism"}
        assert cfg["nx"] * cfg["ny"] * cfg["nz"] == wl.nvox


class FakeNvml:
    """NVML stand-in: a fixed SM clock, and the power-cap reason bit set
    from the third clock query on."""

    def __init__(self, mhz=1965, max_mhz=2070, uuid_ok=True):
        self.mhz, self.max_mhz, self.uuid_ok = mhz, max_mhz, uuid_ok
        self.queries, self.shut = 0, False

    def nvmlInit_v2(self):
        return 0

    def nvmlShutdown(self):
        self.shut = True
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, ref):
        ref._obj.value = 1234
        return 0 if self.uuid_ok and uuid.startswith(b"GPU-") else 13

    def nvmlDeviceGetMaxClockInfo(self, h, kind, ref):
        ref._obj.value = self.max_mhz
        return 0

    def nvmlDeviceGetClockInfo(self, h, kind, ref):
        assert kind == 1
        self.queries += 1
        ref._obj.value = self.mhz
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, ref):
        ref._obj.value = 0x4 | 0x1 if self.queries >= 3 else 0x1
        return 0


def test_nvml_clock_sampler_with_a_stand_in_library():
    import time
    fake = FakeNvml()
    t0 = time.time()
    s = bench.NvmlSampler("GPU-0000", period_s=0.002, lib=fake)
    assert s.ok
    time.sleep(0.05)
    out = s.stop(t0, time.time())
    assert fake.shut and fake.queries >= 3
    assert out["sm_mhz"] == 1965 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] >= 3
    # an unknown device: no sampler (the bench then uses nvidia-smi)
    assert not bench.NvmlSampler("GPU-0000", lib=FakeNvml(uuid_ok=False)).ok
    assert not bench.NvmlSampler(None, lib=FakeNvml()).ok


def test_clock_summary_decodes_the_reason_bits():
    rows = [(1.0, 2070.0, 0x0), (1.1, 2055.0, 0x8), (1.2, 2070.0, 0x40 | 0x20), (5.0, 300.0, 0x4)]
    out = bench.NvmlSampler.summary(rows, 0.9, 1.3, 2070.0, 0.01)
    assert out["sm_mhz"] == 2070.0 and out["samples"] == 3
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert bench.NvmlSampler.summary(rows, 10.0, 11.0, 2070.0, 0.01) is None
