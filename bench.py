#!/usr/bin/env python3
"""Throughput of the fused FGP step on the 3D TV dual, one JSON line.

Workload (default): the 512^3 fp32 volume, 20 outer iterations x 10 FGP steps
with p and r warm-started across outers, t reset to 1 at each outer, fresh
noise in b at each outer, lambda 0.02.  One bench step is one outer
iteration: tvfgp_run (10 FGP steps) + tvfgp_primal (z of p).

Metric: Gvoxel-updates per second (voxels x FGP steps / s), with ms per FGP
step beside it, and the HBM roofline fraction of the step kernel from the
13-volume traffic model of the page "TV solver: the FGP step on the GPU"
(section "Variants": b and the three components of r and of p are read,
p and r written back, 13 fp32 volumes = 52 bytes per voxel and step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Under torchrun with N > 1 each rank runs an independent replica (the step
needs no exchange between replicas): weak scaling, max time over ranks.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ms per FGP step and Gvoxel/s at 512³ fp32; % of GB300 HBM roofline"
UNIT = "Gvoxel/s"
BYTES_PER_VOXEL_STEP = 52        # 13 fp32 volumes per FGP step
BYTES_PER_VOXEL_PRIMAL = 20      # read b, dual(3); write z
# page "TV solver: the FGP step on the GPU", section "At 512³": the fused
# kernel on an RTX 5070, 12.607 ms per FGP step at 512^3
PAGE_FUSED_512_MS = 12.607
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100, help="timed bench steps (outer iterations)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="c4", help="c1..c5 (default c4: 512^3)")
    ap.add_argument("--variant", default="auto", choices=["auto", "fused", "scalar", "zmarch", "zmarch2", "separate", "cube"])
    ap.add_argument("--eager", action="store_true", help="launch eagerly instead of graph replay")
    ap.add_argument("--dual", default="f32", choices=["f32", "f16"],
                    help="storage of p and r (f16: binary16, fp32 arithmetic; changes the result)")
    ap.add_argument("--pitch", default="dense", choices=["dense", "fft"],
                    help="row layout of every volume: dense, or padded to 2*(nx/2+1) floats "
                         "(in-place real-to-complex FFT layout: runs of >= 4 steps are packed into "
                         "dense buffers, shorter ones run in place)")
    ap.add_argument("--b-host", default="wc", choices=["wc", "pinned"],
                    help="page-locked host staging of b for the end-to-end run: write-combined or cached")
    ap.add_argument("--z-host", default="pinned", choices=["wc", "pinned"],
                    help="page-locked host memory receiving z in the end-to-end run: write-combined or cached")
    ap.add_argument("--copy-streams", type=int, default=1,
                    help="end-to-end run: each step's H2D of b and D2H of z split into this many chunks "
                         "along z, each on its own stream (so several copy engines work at once)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-threads", default="",
                    help="comma-separated oracle thread counts for the CPU baseline (default: all cores)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (independent replicas)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world):
    if world <= 1:
        return None
    import torch
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "50"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [s.strip() for s in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.file.name)
        inside = [r for r in rows if t0 - 0.1 <= r[0] <= t1 + 0.1] or rows
        if not inside:
            return None
        reasons = sorted({n for r in inside for n, v in zip(self.NAMES, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "source": "nvidia-smi every 50 ms"}


class NvmlSampler:
    """The SM clock and the active clock-event reasons, read through NVML
    (read-only queries) on a host thread every `period_s` seconds: a short
    timed region still gets a dozen samples or more.  `lib` is the NVML
    library (a stand-in in the host tests).  `ok` is False when NVML or the
    device cannot be opened; the caller then falls back to nvidia-smi."""
    CLOCK_SM = 1                                   # nvmlClockType_t NVML_CLOCK_SM
    BITS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
            ("hw_thermal_slowdown", 0x40))

    def __init__(self, uuid: str | None, period_s: float = 0.01, lib=None):
        import ctypes
        import threading
        self.rows, self.ok, self.period = [], False, period_s
        self.max_mhz = None
        self._ct = ctypes
        try:
            self.lib = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
            if not uuid or self.lib.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
                self.lib.nvmlShutdown()
                return
            self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint(0)
            if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
        except (OSError, AttributeError):
            return
        self.ok = True
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._loop, daemon=True)
        self._thread.start()

    def _loop(self):
        ct = self._ct
        mhz, rs = ct.c_uint(0), ct.c_ulonglong(0)
        while not self._stop.is_set():
            t = time.time()
            if (self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ct.byref(mhz)) == 0
                    and self.reasons_fn(self.h, ct.byref(rs)) == 0):
                self.rows.append((t, float(mhz.value), int(rs.value)))
            self._stop.wait(self.period)

    def stop(self, t0: float, t1: float):
        if not self.ok:
            return None
        self._stop.set()
        self._thread.join(timeout=5)
        self.lib.nvmlShutdown()
        return self.summary(self.rows, t0, t1, self.max_mhz, self.period)

    @classmethod
    def summary(cls, rows, t0: float, t1: float, max_mhz, period_s: float):
        """Median SM clock and the union of the throttle reasons over the
        samples taken inside [t0, t1]."""
        inside = [r for r in rows if t0 <= r[0] <= t1] or [r for r in rows if t0 - 0.1 <= r[0] <= t1 + 0.1]
        if not inside:
            return None
        reasons = sorted({n for r in inside for n, bit in cls.BITS if r[2] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max_mhz if max_mhz is not None else max(r[1] for r in inside),
                "reasons": reasons, "samples": len(inside),
                "source": "NVML every %g ms on a host thread" % (period_s * 1e3)}


def start_clock_sampler(uuid: str | None):
    """NVML sampling when it can be opened, else nvidia-smi every 50 ms."""
    nv = NvmlSampler(uuid)
    return nv if nv.ok else ClockSampler(uuid)


def gpu_id_for(torch, dev) -> str | None:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[0] if vis else None


# ---------------------------------------------------------------------------
# roofline inputs
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _strip_comments(src: str) -> str:
    """C++ source without comments and blank-line differences (string
    literals kept), so that comment edits keep the hash."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (ln.rstrip() for ln in "".join(out).splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash() -> str:
    """Hash of the device code of the step kernels (the headers that hold the
    kernels and their launch shapes), comments excluded; host-only and
    comment-only changes keep it."""
    h = hashlib.sha256()
    for fn in ("fgp_kernels.cuh", "zmarch_tma.cuh", "zmarch2_tma.cuh"):
        with open(os.path.join(ROOT, "fgp_dual_stencil_gb300", "csrc", fn)) as f:
            h.update(_strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_name: str, nvox: int):
    """DRAM bytes per launch of the step kernel from the committed ncu
    summary, scaled to this volume; None when the kernel source changed since
    the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel_name)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return float(ent["dram_bytes_per_voxel"]) * nvox


def roofline_entry(kname, alg_bytes, launch_s, peak, peak_kind, traffic, steps_per_launch, per_voxel_step,
                   f16=False):
    """The bench line's roofline object for the step kernel.  frac: the
    page's traffic model (algorithmic bytes of one launch) over the launch
    time, against the measured copy peak; above 1 when a launch does more
    than one FGP step per pass over memory.  dram_frac: the DRAM bytes ncu
    measured for one launch (traffic) over the same launch time: the share of
    HBM bandwidth the kernel actually draws."""
    achieved = alg_bytes / launch_s / 1e9
    dram = None if traffic is None else traffic / launch_s / 1e9
    return {
        "bound": "hbm",
        "kernel": kname,
        "achieved": round(achieved, 1),
        "peak": peak,
        "unit": "GB/s",
        "frac": round(achieved / peak, 4),
        "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs, copy burst)" % peak_kind
        if peak_kind == "measured" else "fallback 6.8 TB/s",
        "traffic": None if traffic is None else round(traffic),
        "algorithmic_bytes_per_launch": round(alg_bytes),
        "model": ("28 B per voxel and FGP step (b fp32, p and r binary16)" if f16 else
                  "52 B per voxel and FGP step (13 fp32 volumes)") + " x voxel-steps per launch",
        "model_frac": round(achieved / peak, 4),
        "model_frac_basis": "%g FGP step(s) per launch, %d B per voxel and step" % (steps_per_launch, per_voxel_step),
        "dram_achieved": None if dram is None else round(dram, 1),
        "dram_frac": None if dram is None else round(dram / peak, 4),
    }


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def gpu_arm(args, world, rank, local_rank, dist):
    import numpy as np
    import torch
    from fgp_dual_stencil_gb300 import synth
    from fgp_dual_stencil_gb300 import tvfgp as T

    w = synth.WORKLOADS[args.workload]
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    N, K, W = w.nvox, args.steps, args.warmup
    n_b = max(1, min(w.outers, W + K))

    base = synth.phantom(w)
    pitch = T.fft_pitch(w.nx) if args.pitch == "fft" else w.nx
    # inputs staged in the library's write-combined page-locked memory: the
    # GPU reads it at a steady rate (CPU-cached pinned pages on a coherent
    # host showed copy times varying several-fold from copy to copy)
    b_host = []
    for k in range(n_b):
        t = T.host_tensor((w.nz, w.ny, pitch), write_combined=args.b_host == "wc")
        bk = synth.make_b(w, k, base)
        if pitch == w.nx:
            t.numpy()[...] = bk
        else:
            full = np.zeros((w.nz, w.ny, pitch), np.float32)
            full[..., :w.nx] = bk
            t.numpy()[...] = full
        b_host.append(t)
    b_dev = [x.to(dev) for x in b_host]
    shape = (3, w.nz, w.ny, pitch)
    f16 = args.dual == "f16"
    ddt = torch.float16 if f16 else torch.float32
    p = torch.zeros(shape, dtype=ddt, device=dev)
    r = torch.zeros(shape, dtype=ddt, device=dev)
    z = torch.empty((w.nz, w.ny, pitch), device=dev)
    h = T.Tvfgp(w.nx, w.ny, w.nz, args.variant, graph=not args.eager,
                pitch=None if pitch == w.nx else pitch)
    stream = torch.cuda.current_stream(dev)
    run = h.run_f16 if f16 else h.run
    primal = h.primal_f16 if f16 else h.primal

    def outer(b):
        run(b, p, r, w.lam, w.steps, w.t0, stream)
        primal(b, p, w.lam, z, stream)

    for j in range(W):
        outer(b_dev[j % n_b])
    if h.check(stream) != T.TVFGP_OK:
        raise RuntimeError("device error word set during warm-up")
    variant_used = h.last_variant
    launches0 = h.launch_count

    sampler = start_clock_sampler(gpu_id_for(torch, dev)) if not args.no_clocks else None
    if isinstance(sampler, ClockSampler):
        time.sleep(0.6)                       # let nvidia-smi start before the timed region
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    ev_run = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
    barrier(dist)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    ev_start.record(stream)
    for j in range(K):
        b = b_dev[(W + j) % n_b]
        ev_run[j][0].record(stream)
        run(b, p, r, w.lam, w.steps, w.t0, stream)
        ev_run[j][1].record(stream)
        primal(b, p, w.lam, z, stream)
    ev_end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(dist)
    clocks = sampler.stop(t_wall0, t_wall1) if sampler is not None else None
    if h.check(stream) != T.TVFGP_OK:
        raise RuntimeError("device error word set during the timed region")
    launches = h.launch_count - launches0

    elapsed_ms = max_over_ranks(dist, ev_start.elapsed_time(ev_end))
    run_ms = max_over_ranks(dist, sum(a.elapsed_time(b_) for a, b_ in ev_run))
    # step-kernel launches per run: two steps per launch for the two-step
    # kernel (a last odd step runs alone)
    pairs = variant_used == T.TVFGP_VARIANT_ZMARCH2_TMA and w.steps >= 4
    separate = variant_used == T.TVFGP_VARIANT_SEPARATE       # two launches, 18 volumes per step
    launches_per_run = (w.steps // 2 + w.steps % 2) if pairs else (2 * w.steps if separate else w.steps)
    steps_per_launch = w.steps / launches_per_run
    launch_s = run_ms / 1e3 / (K * launches_per_run)
    step_s = run_ms / 1e3 / (K * w.steps)

    value = world * N * w.steps * K / (elapsed_ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()
    # algorithmic bytes: 52 per voxel and FGP step, times the voxel-steps one
    # launch processes
    per_voxel_step = 28 if f16 else (72 if separate else BYTES_PER_VOXEL_STEP)
    alg_bytes = per_voxel_step * N * steps_per_launch
    kname = {T.TVFGP_VARIANT_FUSED: "fgp_step_fused4", T.TVFGP_VARIANT_SCALAR: "fgp_step_scalar",
             T.TVFGP_VARIANT_ZMARCH_TMA: "fgp_step_zmarch_tma",
             T.TVFGP_VARIANT_ZMARCH2_TMA: "fgp_step2_zmarch_tma",
             T.TVFGP_VARIANT_SEPARATE: "primal_vec4 + dual_from_z_vec4",
             T.TVFGP_VARIANT_CUBE_TMA: "fgp_step_cube_tma"}.get(variant_used, "?")
    if f16:
        kname += "<__half>"
    if pitch != w.nx and variant_used == T.TVFGP_VARIANT_FUSED:
        kname = "fgp_step_fused4 (quads as two float2)" if w.nx % 4 == 0 else "fgp_step_fused2"
    traffic = ncu_traffic(kname, N)             # DRAM bytes per launch (ncu), or None

    # end to end: every step's b copied in from pinned host memory and its z
    # copied back, through the public API; the copies run on their own
    # streams (double-buffered) and overlap the previous / next step's compute
    e2e = None
    if not args.no_e2e:
        e2e_s = end_to_end(torch, h, w, b_host, p, r, stream, dev, K, dist, run, primal,
                           z_wc=args.z_host == "wc", copy_streams=args.copy_streams)
        e2e = {"value": round(world * N * w.steps * K / e2e_s / 1e9, 3), "unit": UNIT,
               "h2d_bytes_per_step": 4 * w.ny * w.nz * pitch, "d2h_bytes_per_step": 4 * w.ny * w.nz * pitch,
               "ms_per_step": round(e2e_s * 1e3 / K, 4),
               "overlap": "H2D of step j+1 and D2H of step j, each split along z into %d chunks on %d "
                          "streams, double-buffered" % (args.copy_streams, args.copy_streams),
               "host_memory": "b from %s, z to %s page-locked memory (tvfgp_host_alloc)"
                              % ("write-combined" if args.b_host == "wc" else "cached",
                                 "write-combined" if args.z_host == "wc" else "cached")}
        if h.check(stream) != T.TVFGP_OK:
            raise RuntimeError("device error word set during the end-to-end run")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = [int(t) for t in args.cpu_threads.split(",") if t.strip()]
        cpu = cpu_baseline(w, base, threads)

    h.close()
    names = {T.TVFGP_VARIANT_FUSED: "fused", T.TVFGP_VARIANT_SCALAR: "scalar",
             T.TVFGP_VARIANT_ZMARCH_TMA: "zmarch", T.TVFGP_VARIANT_ZMARCH2_TMA: "zmarch2",
             T.TVFGP_VARIANT_SEPARATE: "separate", T.TVFGP_VARIANT_CUBE_TMA: "cube"}
    out = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(elapsed_ms / K, 4),
        "ms_per_fgp_step": round(elapsed_ms / K / w.steps, 4),
        "ms_per_fgp_step_kernel": round(step_s * 1e3, 4),
        "ms_per_step_launch": round(launch_s * 1e3, 4),
        "fgp_steps_per_launch": steps_per_launch,
        "higher_is_better": True,
        "scaling": "weak",
        # the page's figure is for the fp32 dual at 512^3: no ratio for a
        # binary16 dual (a different result) or another volume
        "vs_baseline": round(value / (N / (PAGE_FUSED_512_MS / 1e3) / 1e9), 3)
        if args.workload == "c4" and not f16 else None,
        "dtype": "f32 (dual stored as f16)" if f16 else "f32",
        "data": "synthetic",
        "config": workload_config(w, world),
        # how this arm ran the workload; kept out of "config" so that both
        # arms describe the same workload with the same dictionary
        "impl_config": {
            "variant": names.get(variant_used, str(variant_used)),
            "launch": "eager" if args.eager else "cuda_graph",
            "row_pitch": pitch,
            "vs_baseline_ref": "RTX 5070 fused kernel, 12.607 ms per FGP step at 512^3 (page figure; "
                               "other hardware, context only)",
        },
        "roofline": roofline_entry(kname, alg_bytes, launch_s, peak, peak_kind, traffic, steps_per_launch,
                                   per_voxel_step, f16),
        "gpu_launches": launches,
        "e2e": e2e,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    return out


def end_to_end(torch, h, w, b_host, p, r, stream, dev, K, dist, run, primal, z_wc=False, copy_streams=4):
    """Wall time of K outer iterations where each step's b comes from pinned
    host memory and its z goes back to pinned host memory.  Each copy is
    split along z into copy_streams chunks, one stream per chunk, so that
    several copy engines move it at once; compute waits for all chunks of its
    b, and z's chunks wait for the step that wrote z."""
    n_b = len(b_host)
    shape = tuple(b_host[0].shape)
    C = max(1, min(int(copy_streams), shape[0]))
    cuts = [shape[0] * c // C for c in range(C + 1)]
    b_in = [torch.empty(shape, device=dev) for _ in range(2)]
    z_out = [torch.empty(shape, device=dev) for _ in range(2)]
    from fgp_dual_stencil_gb300 import tvfgp as T
    z_host = [T.host_tensor(shape, write_combined=z_wc) for _ in range(2)]
    s_in = [torch.cuda.Stream(dev) for _ in range(C)]
    s_out = [torch.cuda.Stream(dev) for _ in range(C)]
    ev_in = [[torch.cuda.Event() for _ in range(C)] for _ in range(2)]    # b_in[s] chunk filled
    ev_done = [torch.cuda.Event() for _ in range(2)]                       # step using slot s finished
    ev_out = [[torch.cuda.Event() for _ in range(C)] for _ in range(2)]   # z_host[s] chunk filled

    def h2d(j):
        s = j % 2
        for c in range(C):
            lo, hi = cuts[c], cuts[c + 1]
            with torch.cuda.stream(s_in[c]):
                if j >= 2:
                    s_in[c].wait_event(ev_done[s])           # b_in[s] no longer read
                b_in[s][lo:hi].copy_(b_host[j % n_b][lo:hi], non_blocking=True)
                ev_in[s][c].record(s_in[c])

    barrier(dist)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    h2d(0)
    for j in range(K):
        s = j % 2
        if j + 1 < K:
            h2d(j + 1)
        for c in range(C):
            stream.wait_event(ev_in[s][c])
            if j >= 2:
                stream.wait_event(ev_out[s][c])              # z_out[s] copied out
        run(b_in[s], p, r, w.lam, w.steps, w.t0, stream)
        primal(b_in[s], p, w.lam, z_out[s], stream)
        ev_done[s].record(stream)
        for c in range(C):
            lo, hi = cuts[c], cuts[c + 1]
            with torch.cuda.stream(s_out[c]):
                s_out[c].wait_event(ev_done[s])
                z_host[s][lo:hi].copy_(z_out[s][lo:hi], non_blocking=True)
                ev_out[s][c].record(s_out[c])
    torch.cuda.synchronize(dev)
    dt = max_over_ranks(dist, time.perf_counter() - t0)
    barrier(dist)
    return dt


def cpu_baseline(w, base, threads=(), budget_s=10.0):
    """The CPU oracle, as it stands, on a bounded sample of the workload, in
    the workload's own order: outer iterations on the full volume (fresh b,
    t reset, p and r carried over), each run in chunks of up to 10 FGP steps
    (momentum carried from chunk to chunk) and ended by the primal, until
    about budget_s seconds of oracle time or the end of the workload.  All
    host cores unless thread counts are given (the first count then gives
    `value`, each count its own entry in `by_threads`).  Making each outer's
    b is not timed."""
    import numpy as np
    import oracle
    from fgp_dual_stencil_gb300 import synth
    all_cores = oracle.get_threads()
    counts = list(threads) or [all_cores]
    res = {}
    b_cur = {}
    for n in counts:
        oracle.set_threads(n)
        p = np.zeros((3, w.nz, w.ny, w.nx), np.float32)
        r = np.zeros_like(p)
        spent, outers, steps = 0.0, 0, 0
        while outers < w.outers and (steps == 0 or spent < budget_s):
            if b_cur.get("k") != outers:
                b_cur = {"k": outers, "b": synth.make_b(w, outers, base)}
            b = b_cur["b"]
            t, done = w.t0, 0
            while done < w.steps and (steps == 0 or spent < budget_s):
                chunk = min(10, w.steps - done)
                t0 = time.perf_counter()
                t = oracle.fgp_run(b, p, r, w.lam, chunk, t)
                spent += time.perf_counter() - t0
                done += chunk
                steps += chunk
            t0 = time.perf_counter()
            oracle.primal(b, p, w.lam)
            spent += time.perf_counter() - t0
            outers += 1
        res[n] = (spent, steps, outers)
    oracle.set_threads(all_cores)
    n0 = counts[0]
    t, k, o = res[n0]
    out = {"value": round(w.nvox * k / t / 1e9, 4), "unit": UNIT, "cores": n0,
           "kind": "oracle",
           "sample": "the first %d FGP steps of the workload (%d outer iteration(s), each ended by the "
                     "primal) on the full %dx%dx%d volume, %.1f s of oracle time"
                     % (k, o, w.nx, w.ny, w.nz, t)}
    if len(counts) > 1:
        out["by_threads"] = {str(n): {"value": round(w.nvox * kk / tt / 1e9, 4),
                                      "ms_per_fgp_step": round(tt * 1e3 / kk, 2),
                                      "fgp_steps": kk} for n, (tt, kk, oo) in res.items()}
    return out


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle on the same workload
# ---------------------------------------------------------------------------

def workload_config(w, world):
    """The bench line's "config": the workload alone, identical for the
    library's arm and the oracle's, so that their lines compare."""
    n = w.nvox
    return {
        "workload": "%dx%dx%d fp32 TV-dual FGP, %d outers x %d steps, warm p/r, t0=1 per outer, "
                    "lambda %g; one bench step = one outer (%d FGP steps + primal)"
                    % (w.nx, w.ny, w.nz, w.outers, w.steps, w.lam, w.steps),
        "nx": w.nx, "ny": w.ny, "nz": w.nz, "fgp_steps_per_bench_step": w.steps,
        "l2": "inputs larger than L2 (%.1f GB of live buffers vs 126 MB L2)" % (11 * 4 * n / 1e9)
        if 4 * n > 129e6 else "working set fits in L2: GB/s is not an HBM figure",
        "parallelism": "replicas" if world > 1 else "single_gpu",
    }


def reference_arm(args, world, rank):
    """The CPU oracle, as it stands, on the GPU arm's workload and metric:
    each bench step is one outer iteration on the full volume (a fresh b, t
    reset to t0, p and r carried over, the workload's FGP steps, then the
    primal).  Making b is not timed."""
    import numpy as np
    import oracle
    from fgp_dual_stencil_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    base = synth.phantom(w)
    n_b = max(1, min(w.outers, W + K))
    bs = {}

    def b_of(j):
        k = j % n_b
        if k not in bs:
            bs[k] = synth.make_b(w, k, base)
        return bs[k]

    p = np.zeros((3, w.nz, w.ny, w.nx), np.float32)
    r = np.zeros_like(p)

    def outer(b):
        t0 = time.perf_counter()
        oracle.fgp_run(b, p, r, w.lam, w.steps, w.t0)
        oracle.primal(b, p, w.lam)
        return time.perf_counter() - t0

    for j in range(W):
        outer(b_of(j))
    dt = sum(outer(b_of(W + j)) for j in range(K))
    value = w.nvox * w.steps * K / dt / 1e9
    sample = ("%d bench steps, each one outer iteration (%d FGP steps + primal) on the full %dx%dx%d volume"
              % (K, w.steps, w.nx, w.ny, w.nz))
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(dt * 1e3 / K, 3),
        "ms_per_fgp_step": round(dt * 1e3 / K / w.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(w, world),
        "impl_config": {"variant": "oracle (plain C, fp64 schedule, fp32 arithmetic)", "launch": "host threads"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": oracle.get_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    args = parse_args()
    world, rank, local_rank = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(reference_arm(args, world, rank)), flush=True)
        return 0
    dist = dist_init(world)
    out = gpu_arm(args, world, rank, local_rank, dist)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
