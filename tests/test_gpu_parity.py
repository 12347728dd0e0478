"""GPU path against the CPU oracle, element by element, on the same seeded
inputs (page "TV solver: the FGP step on the GPU", section "What one step
does").  The bar is max abs diff <= 1e-5 on p and r and <= 1e-5 * max|b| on
z; the kernels evaluate the same canonical fp32 expression order as the
oracle, so the small cases are also checked for exact equality."""
import numpy as np
import pytest

import oracle
from fgp_dual_stencil_gb300 import synth
from gpu_util import (assert_parity, dev, host, max_diff, run_workload_gpu, run_workload_oracle)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available()
    from fgp_dual_stencil_gb300 import tvfgp
    return tvfgp


VEC_VARIANTS = ["fused", "zmarch", "zmarch2", "scalar", "separate", "cube"]


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("variant", VEC_VARIANTS)
@pytest.mark.parametrize("key", ["c1", "c2"])
def test_small_workloads_exact(T, key, variant):
    w = synth.WORKLOADS[key]
    b, *gpu, launched = run_workload_gpu(w, variant)
    ref = run_workload_oracle(w)
    assert_parity(gpu, ref[1:], float(np.abs(b).max()), exact=True, what=key)
    per_outer = w.steps // 2 + w.steps % 2 if (variant == "zmarch2" and w.steps >= 4) else w.steps
    if variant == "separate":
        per_outer = 2 * w.steps
    assert launched == w.outers * per_outer + 2


@pytest.mark.parametrize("variant", ["auto", "cube", "zmarch", "fused", "separate", "scalar"])
def test_256_warm_started_outers_graph(T, variant):
    """20 outers x 10 steps, fresh noise per outer, t0 reset, graph replay
    re-parameterised with every new b."""
    w = synth.WORKLOADS["c3"]
    b, *gpu, _ = run_workload_gpu(w, variant, graph=True)
    ref = run_workload_oracle(w)
    assert_parity(gpu, ref[1:], float(np.abs(b).max()), exact=True, what="c3")


@pytest.mark.slow
@pytest.mark.parametrize("key,variant", [("c4", "auto"), ("c5", "auto"), ("c4", "zmarch2"), ("c4", "cube"),
                                         ("c5", "zmarch")])
def test_large_workloads(T, key, variant):
    """The 512^3 workload and the 1000x600x300 blob volume in the
    configuration the bench times (AUTO variant, graph replay), and again
    with other kernels (two steps per launch, cube tiles, one step per
    launch)."""
    w = synth.WORKLOADS[key]
    b, *gpu, _ = run_workload_gpu(w, variant, graph=(key == "c4" or variant == "auto"))
    ref = run_workload_oracle(w)
    assert_parity(gpu, ref[1:], float(np.abs(b).max()), exact=False, what=key)
    # the result is still checked for exact equality, reported separately
    assert max_diff(gpu[0], ref[1]) == 0.0 and max_diff(gpu[1], ref[2]) == 0.0


# ---------------------------------------------------------------------------
# shapes, ragged tails, step counts, warm starts
# ---------------------------------------------------------------------------

ODD_SHAPES = [(1, 1, 1), (2, 1, 1), (1, 2, 1), (1, 1, 2), (5, 3, 7), (33, 17, 9), (4, 1, 1),
              (8, 3, 2), (132, 9, 11), (260, 5, 19), (36, 40, 3), (1, 64, 64)]


@pytest.mark.parametrize("shape", ODD_SHAPES)
@pytest.mark.parametrize("variant", VEC_VARIANTS)
def test_odd_shapes_warm_start(T, shape, variant):
    nx, ny, nz = shape
    seed = nx * 1000 + ny * 10 + nz
    b = synth.random_case(shape, seed)
    p0 = synth.random_dual(shape, seed, scale=0.4)
    r0 = synth.random_dual(shape, seed + 1, scale=0.6)
    lam = 0.07
    for nsteps in ((0, 1, 2, 3, 4, 5, 6, 7, 10) if variant == "zmarch2" else (0, 1, 2, 3, 7)):
        p, r = dev(p0), dev(r0)
        bd = dev(b)
        with T.Tvfgp(nx, ny, nz, variant) as h:
            tf = h.run(bd, p, r, lam, nsteps, 1.0)
            zp = h.primal(bd, p, lam)
            assert h.check() == 0
            if nsteps:
                if variant == "separate":
                    want = T.TVFGP_VARIANT_SEPARATE
                elif variant == "scalar" or nx % 4:
                    want = T.TVFGP_VARIANT_SCALAR
                elif variant == "zmarch2" and nsteps < 4:
                    want = T.TVFGP_VARIANT_ZMARCH_TMA      # two-step launches from 4 steps on
                else:
                    want = T.VARIANTS[variant]
                assert h.last_variant == want
        po, ro = p0.copy(), r0.copy()
        tfo = oracle.fgp_run(b, po, ro, lam, nsteps, 1.0)
        assert tf == tfo
        assert max_diff(host(p), po) == 0.0, (shape, nsteps, "p")
        assert max_diff(host(r), ro) == 0.0, (shape, nsteps, "r")
        assert max_diff(host(zp), oracle.primal(b, po, lam)) == 0.0, (shape, nsteps, "z")


def test_continuing_a_run_with_t_final(T):
    """Two runs chained through t_final equal one long run."""
    w = synth.WORKLOADS["c1"]
    b = dev(synth.make_b(w, 0))
    shape = (3, w.nz, w.ny, w.nx)
    import torch
    p1, r1 = torch.zeros(shape, device="cuda"), torch.zeros(shape, device="cuda")
    p2, r2 = torch.zeros(shape, device="cuda"), torch.zeros(shape, device="cuda")
    with T.Tvfgp(w.nx, w.ny, w.nz) as h:
        h.run(b, p1, r1, w.lam, 17, 1.0)
        t = h.run(b, p2, r2, w.lam, 6, 1.0)
        h.run(b, p2, r2, w.lam, 11, t)
    assert torch.equal(p1, p2) and torch.equal(r1, r2)


def test_upper_faces_stay_zero(T):
    w = synth.WORKLOADS["c2"]
    _, p, r, _, _, _ = run_workload_gpu(w, "fused")
    for f in (p, r):
        assert not f[0][:, :, -1].any() and not f[1][:, -1, :].any() and not f[2][-1].any()
    assert np.sqrt((p.astype(np.float64) ** 2).sum(0)).max() <= 1 + 2 ** -22


# ---------------------------------------------------------------------------
# entry points: step, primal, graph, variants, fallbacks
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(64, 32, 16), (30, 7, 5)])
def test_step_entry_matches_oracle_step(T, shape):
    nx, ny, nz = shape
    b = synth.random_case(shape, 3)
    p0 = synth.random_dual(shape, 4)
    rs = synth.random_dual(shape, 5, scale=0.8)
    lam, m = 0.05, np.float32(0.37)
    p, rsd, rdd = dev(p0), dev(rs), dev(np.zeros_like(rs))
    with T.Tvfgp(nx, ny, nz) as h:
        h.step(dev(b), p, rsd, rdd, lam, float(m))
        h.check()
    po = p0.copy()
    rdo, _ = oracle.fgp_step(b, po, rs, np.float32(lam), m)
    assert max_diff(host(p), po) == 0.0 and max_diff(host(rdd), rdo) == 0.0
    assert max_diff(host(rsd), rs) == 0.0          # r_src is not written


def test_graph_equals_eager_and_reparameterises(T):
    import torch
    w = synth.WORKLOADS["c2"]
    base = synth.phantom(w)
    bs = [dev(synth.make_b(w, k, base)) for k in range(3)]
    shape = (3, w.nz, w.ny, w.nx)
    out = {}
    for graph in (False, True):
        p, r = torch.zeros(shape, device="cuda"), torch.zeros(shape, device="cuda")
        with T.Tvfgp(w.nx, w.ny, w.nz, "auto", graph) as h:
            t = 1.0
            for k, nsteps in enumerate((10, 10, 5, 10, 5)):
                # new b, t0 and step count each call: rebuild / re-parameterise
                t = h.run(bs[k % 3], p, r, w.lam * (1 + 0.1 * k), nsteps, 1.0 if k % 2 == 0 else t)
            h.check()
        out[graph] = (p, r)
    assert torch.equal(out[False][0], out[True][0]) and torch.equal(out[False][1], out[True][1])


def test_variants_agree_bitwise(T):
    import torch
    w = synth.WORKLOADS["c2"]
    res = []
    for v in VEC_VARIANTS:
        _, p, r, zp, _, _ = run_workload_gpu(w, v)
        res.append((p, r, zp))
    for other in res[1:]:
        for a, b in zip(res[0], other):
            assert np.array_equal(a, b)


def test_misaligned_pointers_fall_back_to_scalar(T):
    import torch
    nx, ny, nz = 16, 8, 4
    n = nx * ny * nz
    b = synth.random_case((nx, ny, nz), 9)
    p0 = synth.random_dual((nx, ny, nz), 10)
    r0 = synth.random_dual((nx, ny, nz), 11)
    # 4-byte aligned but not 16-byte aligned views
    bb = torch.zeros(n + 1, device="cuda"); bb[1:] = dev(b).view(-1)
    pb = torch.zeros(3 * n + 1, device="cuda"); pb[1:] = dev(p0).view(-1)
    rb = torch.zeros(3 * n + 1, device="cuda"); rb[1:] = dev(r0).view(-1)
    with T.Tvfgp(nx, ny, nz) as h:
        h.run(bb[1:], pb[1:], rb[1:], 0.05, 4, 1.0)
        assert h.last_variant == T.TVFGP_VARIANT_SCALAR
        h.check()
    po, ro = p0.copy(), r0.copy()
    oracle.fgp_run(b, po, ro, 0.05, 4, 1.0)
    assert max_diff(host(pb[1:]).reshape(po.shape), po) == 0.0
    assert max_diff(host(rb[1:]).reshape(ro.shape), ro) == 0.0


# ---------------------------------------------------------------------------
# argument errors and the bounded-wait error path
# ---------------------------------------------------------------------------

def test_argument_errors_enqueue_nothing(T):
    import ctypes
    import torch
    nx, ny, nz = 8, 4, 4
    n = nx * ny * nz
    b = torch.rand(n, device="cuda")
    p = torch.rand(3 * n, device="cuda")
    r = torch.rand(3 * n, device="cuda")
    p_keep, r_keep = p.clone(), r.clone()
    h = T.tvfgp_create(nx, ny, nz)
    try:
        B, P, R = b.data_ptr(), p.data_ptr(), r.data_ptr()
        tf = ctypes.c_double()
        run = lambda *a: T.raw_call("tvfgp_run", h, *a, None, ctypes.byref(tf))
        assert run(B, P, R, 0.0, 3, 1.0) == T.TVFGP_ERR_ARG
        assert run(B, P, R, -1.0, 3, 1.0) == T.TVFGP_ERR_ARG
        assert run(B, P, R, float("nan"), 3, 1.0) == T.TVFGP_ERR_ARG
        assert run(B, P, R, float("inf"), 3, 1.0) == T.TVFGP_ERR_ARG
        assert run(B, P, R, 1e-45, 3, 1.0) == T.TVFGP_ERR_ARG          # 1/(12 lambda) overflows
        assert run(B, P, R, 0.1, -1, 1.0) == T.TVFGP_ERR_ARG
        assert run(B, P, R, 0.1, 3, 0.5) == T.TVFGP_ERR_ARG
        assert run(None, P, R, 0.1, 3, 1.0) == T.TVFGP_ERR_ARG
        assert run(B + 2, P, R, 0.1, 3, 1.0) == T.TVFGP_ERR_ALIGN
        assert run(B, P, P, 0.1, 3, 1.0) == T.TVFGP_ERR_ARG            # p and r alias
        assert T.raw_call("tvfgp_run", None, B, P, R, 0.1, 3, 1.0, None, None) == T.TVFGP_ERR_ARG
        assert T.raw_call("tvfgp_step", h, B, P, R, R, ctypes.c_float(0.1), ctypes.c_float(0.2), None) == T.TVFGP_ERR_ARG
        assert T.raw_call("tvfgp_primal", h, B, P, ctypes.c_float(0.1), B, None) == T.TVFGP_ERR_ARG
        assert T.raw_call("tvfgp_set_variant", h, 9) == T.TVFGP_ERR_ARG
        assert T.tvfgp_launch_count(h) == 0
        torch.cuda.synchronize()
        assert torch.equal(p, p_keep) and torch.equal(r, r_keep)
        assert T.tvfgp_check(h) == T.TVFGP_OK
    finally:
        T.tvfgp_destroy(h)


def test_bounded_wait_reports_timeout_and_context_survives(T):
    import torch
    w = synth.WORKLOADS["c1"]
    with T.Tvfgp(w.nx, w.ny, w.nz) as h:
        T.tvfgp_debug_timeout_probe(h.h, 2000)
        assert h.check() == T.TVFGP_ERR_TIMEOUT
        assert h.check() == T.TVFGP_OK            # the error word was cleared
        b = dev(synth.make_b(w, 0))
        p = torch.zeros((3, w.nz, w.ny, w.nx), device="cuda")
        r = torch.zeros_like(p)
        h.run(b, p, r, w.lam, w.steps, 1.0)
        assert h.check() == T.TVFGP_OK
    po = np.zeros_like(host(p)); ro = np.zeros_like(po)
    oracle.fgp_run(synth.make_b(w, 0), po, ro, w.lam, w.steps, 1.0)
    assert max_diff(host(p), po) == 0.0


@pytest.mark.parametrize("variant,steps,f16,from_plane", [
    ("zmarch2", 6, False, 0), ("zmarch2", 5, False, 0), ("zmarch2", 6, False, 4), ("zmarch2", 4, False, 6),
    ("zmarch", 3, False, 0), ("zmarch", 3, False, 5), ("cube", 3, False, 0), ("auto", 4, True, 0),
    ("auto", 4, True, 3)])
def test_step_kernels_own_timeout_path(T, variant, steps, f16, from_plane):
    """With a poll limit of 0 every CTA of the TMA kernels gives up at its
    first wait for data of plane from_plane or later (the first wait, or in
    the middle of the march with copies of later planes in flight): it must
    record the timeout, wait for its copies in flight and return, leaving the
    context usable; with the default limit restored the same handle runs bit
    for bit as the oracle."""
    import torch
    shape = (72, 40, 37)
    nx, ny, nz = shape
    lam = 0.06
    b = synth.random_case(shape, 71)
    p0 = synth.random_dual(shape, 72, scale=0.4)
    r0 = synth.random_dual(shape, 73, scale=0.6)
    if f16:
        p0, r0 = oracle.float_to_half(p0), oracle.float_to_half(r0)

    def fresh():
        if f16:
            return (torch.from_numpy(p0.view(np.float16)).cuda(), torch.from_numpy(r0.view(np.float16)).cuda())
        return dev(p0), dev(r0)

    bd = dev(b)
    with T.Tvfgp(nx, ny, nz, variant) as h:
        run = h.run_f16 if f16 else h.run
        T.tvfgp_debug_set_poll_limit(h.h, 0, from_plane)
        p, r = fresh()
        run(bd, p, r, lam, steps, 1.0)
        assert h.check() == T.TVFGP_ERR_TIMEOUT
        assert h.check() == T.TVFGP_OK
        T.tvfgp_debug_set_poll_limit(h.h, -1)
        p, r = fresh()
        run(bd, p, r, lam, steps, 1.0)
        assert h.check() == T.TVFGP_OK
        used = h.last_variant
    want = {"zmarch2": (T.TVFGP_VARIANT_ZMARCH2_TMA, T.TVFGP_VARIANT_ZMARCH_TMA),
            "zmarch": (T.TVFGP_VARIANT_ZMARCH_TMA,), "cube": (T.TVFGP_VARIANT_CUBE_TMA,),
            "auto": (T.TVFGP_VARIANT_ZMARCH_TMA,)}[variant]
    assert used in want, used
    po, ro = p0.copy(), r0.copy()
    if f16:
        oracle.fgp_run_h16(b, po, ro, lam, steps, 1.0)
        assert np.array_equal(p.cpu().numpy().view(np.uint16), po)
        assert np.array_equal(r.cpu().numpy().view(np.uint16), ro)
    else:
        oracle.fgp_run(b, po, ro, lam, steps, 1.0)
        assert np.array_equal(host(p), po) and np.array_equal(host(r), ro)


def test_poll_limit_arguments(T):
    with T.Tvfgp(8, 4, 4) as h:
        assert T.raw_call("tvfgp_debug_set_poll_limit", h.h, (1 << 22) + 1, 0) == T.TVFGP_ERR_ARG
        assert T.raw_call("tvfgp_debug_set_poll_limit", h.h, 0, -1) == T.TVFGP_ERR_ARG
        assert T.raw_call("tvfgp_debug_set_poll_limit", None, 0, 0) == T.TVFGP_ERR_ARG
        assert T.raw_call("tvfgp_debug_set_poll_limit", h.h, 1 << 22, 3) == T.TVFGP_OK
        assert T.raw_call("tvfgp_debug_set_poll_limit", h.h, -1, 0) == T.TVFGP_OK


@pytest.mark.parametrize("wc", [False, True])
def test_host_staging_memory_round_trip(T, wc):
    """Pinned (and write-combined) host memory from the library as the source
    of an input copy and the target of a result copy."""
    import torch
    torch.zeros(1, device="cuda")          # torch reports pinning only once CUDA is up
    shape = (33, 17, 9)
    src = T.host_tensor((shape[2], shape[1], shape[0]), write_combined=wc)
    assert src.is_pinned()
    b = synth.random_case(shape, 5)
    src.numpy()[...] = b
    d = torch.empty_like(src, device="cuda")
    d.copy_(src, non_blocking=True)
    out = T.host_tensor(src.shape, write_combined=False)
    out.copy_(d * 2, non_blocking=True)
    torch.cuda.synchronize()
    assert np.array_equal(out.numpy(), 2 * b)


# ---------------------------------------------------------------------------
# seeded random shapes: tile, chunk and tail boundaries anywhere
# ---------------------------------------------------------------------------

def random_shapes(count, seed):
    """Shapes drawn so that x is a multiple of 4 in most cases (the vector
    and TMA kernels) and not in the rest (the scalar fallback), with y and
    z anywhere from one plane to several tiles and chunks."""
    rng = np.random.default_rng(seed)
    out = []
    for k in range(count):
        nx = int(rng.integers(1, 50)) * 4 if k % 4 else int(rng.integers(1, 200))
        ny = int(rng.integers(1, 90))
        nz = int(rng.integers(1, 160))
        out.append((nx, ny, nz))
    return out


@pytest.mark.parametrize("shape", random_shapes(12, 20261202))
@pytest.mark.parametrize("variant", ["auto", "zmarch2", "zmarch", "cube"])
def test_random_shapes_match_the_oracle(T, shape, variant):
    nx, ny, nz = shape
    seed = (nx * 131 + ny) * 197 + nz
    rng = np.random.default_rng(seed)
    nsteps = int(rng.integers(4, 10))
    lam = float(rng.uniform(0.01, 0.2))
    b = synth.random_case(shape, seed)
    p0 = synth.random_dual(shape, seed + 1, scale=0.5)
    r0 = synth.random_dual(shape, seed + 2, scale=0.7)
    p, r, bd = dev(p0), dev(r0), dev(b)
    with T.Tvfgp(nx, ny, nz, variant) as h:
        tf = h.run(bd, p, r, lam, nsteps, 1.0)
        zp = h.primal(bd, p, lam)
        assert h.check() == 0
    po, ro = p0.copy(), r0.copy()
    assert tf == oracle.fgp_run(b, po, ro, lam, nsteps, 1.0)
    assert max_diff(host(p), po) == 0.0, (shape, variant, nsteps, lam, "p")
    assert max_diff(host(r), ro) == 0.0, (shape, variant, nsteps, lam, "r")
    assert max_diff(host(zp), oracle.primal(b, po, lam)) == 0.0, (shape, variant, nsteps, lam, "z")
