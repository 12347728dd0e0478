"""The dual stored in half precision (tvfgp_run_f16 / tvfgp_primal_f16)
against the CPU oracle with the same storage: exact equality, and the
measured accuracy against the fp32 result."""
import numpy as np
import pytest

import oracle
from fgp_dual_stencil_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available()
    from fgp_dual_stencil_gb300 import tvfgp
    return tvfgp


def dev16(a16):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a16).view(np.float16)).cuda()


def bits(t):
    return t.detach().cpu().numpy().view(np.uint16)


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("key", ["c1", "c2"])
def test_workloads_exact(T, key, graph):
    w = synth.WORKLOADS[key]
    b = synth.make_b(w, 0)
    shape = (3,) + b.shape
    ph = np.zeros(shape, np.uint16)
    rh = np.zeros(shape, np.uint16)
    p, r = dev16(ph), dev16(rh)
    bd = dev(b)
    with T.Tvfgp(w.nx, w.ny, w.nz, "auto", graph) as h:
        h.run_f16(bd, p, r, w.lam, w.steps, 1.0)
        z = h.primal_f16(bd, p, w.lam)
        assert h.check() == 0
    oracle.fgp_run_h16(b, ph, rh, w.lam, w.steps, 1.0)
    assert np.array_equal(bits(p), ph) and np.array_equal(bits(r), rh)
    assert np.array_equal(z.cpu().numpy(), oracle.primal_h16(b, ph, w.lam))


F16_SHAPES = [(1, 1, 1), (5, 3, 7), (33, 17, 9), (36, 40, 3), (132, 9, 11),
              (8, 1, 1), (8, 3, 2), (40, 17, 9), (72, 31, 37), (264, 5, 19), (16, 64, 64)]


def expected_variant(T, nx, variant):
    """The kernel run_f16 picks: the z-march when rows are whole 16-byte
    units (nx % 8 == 0), else the fused kernel when nx % 4 == 0, else the
    scalar one; FUSED and SCALAR handles keep to their own kernel."""
    if variant == "scalar":
        return T.TVFGP_VARIANT_SCALAR
    if nx % 8 == 0 and variant != "fused":
        return T.TVFGP_VARIANT_ZMARCH_TMA
    return T.TVFGP_VARIANT_FUSED if nx % 4 == 0 else T.TVFGP_VARIANT_SCALAR


@pytest.mark.parametrize("shape", F16_SHAPES)
def test_odd_shapes_exact(T, shape):
    nx, ny, nz = shape
    b = synth.random_case(shape, 31)
    p0 = oracle.float_to_half(synth.random_dual(shape, 32, scale=0.4))
    r0 = oracle.float_to_half(synth.random_dual(shape, 33, scale=0.6))
    for nsteps in (0, 1, 2, 3, 7):
        p, r = dev16(p0), dev16(r0)
        with T.Tvfgp(nx, ny, nz) as h:
            h.run_f16(dev(b), p, r, 0.07, nsteps, 1.0)
            assert h.last_variant == expected_variant(T, nx, "auto") or nsteps == 0
            assert h.check() == 0
        ph, rh = p0.copy(), r0.copy()
        oracle.fgp_run_h16(b, ph, rh, 0.07, nsteps, 1.0)
        assert np.array_equal(bits(p), ph), (shape, nsteps)
        assert np.array_equal(bits(r), rh), (shape, nsteps)


@pytest.mark.parametrize("variant", ["auto", "fused", "scalar"])
def test_f16_kernels_agree_bitwise(T, variant):
    """The three binary16 kernels on a volume where all three can run (64 x
    45 x 40: several tiles in x and y, ragged in y, several march segments
    in z) give the oracle's bits, eager and through a graph."""
    shape = (64, 45, 40)
    b = synth.random_case(shape, 41)
    p0 = oracle.float_to_half(synth.random_dual(shape, 42, scale=0.5))
    r0 = oracle.float_to_half(synth.random_dual(shape, 43, scale=0.7))
    ph, rh = p0.copy(), r0.copy()
    oracle.fgp_run_h16(b, ph, rh, 0.05, 5, 1.0)
    for graph in (False, True):
        p, r = dev16(p0), dev16(r0)
        with T.Tvfgp(*shape, variant, graph) as h:
            h.run_f16(dev(b), p, r, 0.05, 5, 1.0)
            assert h.last_variant == expected_variant(T, shape[0], variant)
            assert h.check() == 0
        assert np.array_equal(bits(p), ph) and np.array_equal(bits(r), rh), (variant, graph)


@pytest.mark.parametrize("variant", ["auto", "fused", "scalar"])
@pytest.mark.parametrize("lam", [0.05, 1e-17, 1e4])
def test_f16_subnormal_and_extreme_codes(T, variant, lam):
    """Stored duals drawn from every binary16 subnormal code, both signed
    zeros, +-1, the smallest normal and +-65504, with half of b negative (z
    clamps to 0) and the rest tiny; the results are full of binary16
    subnormals.  lam = 1e-17 sends the projection to its IEEE fallback."""
    shape = (48, 13, 9)
    nx, ny, nz = shape
    g = np.random.default_rng(7)
    sub = np.arange(1, 1024, dtype=np.uint16)
    codes = np.concatenate([sub, sub | 0x8000, np.uint16([0x7bff, 0xfbff, 0x3c00, 0xbc00, 0x0400, 0x8400, 0, 0x8000])])
    p0 = g.choice(codes, size=(3, nz, ny, nx)).astype(np.uint16)
    r0 = g.choice(codes, size=(3, nz, ny, nx)).astype(np.uint16)
    b = np.where(g.uniform(size=(nz, ny, nx)) < 0.5, -1.0, g.uniform(0, 1e-4, (nz, ny, nx))).astype(np.float32)
    ph, rh = p0.copy(), r0.copy()
    oracle.fgp_run_h16(b, ph, rh, lam, 5, 1.0)
    p, r = dev16(p0), dev16(r0)
    with T.Tvfgp(*shape, variant) as h:
        h.run_f16(dev(b), p, r, lam, 5, 1.0)
        z = h.primal_f16(dev(b), p, lam)
        assert h.check() == 0
    assert np.array_equal(bits(p), ph) and np.array_equal(bits(r), rh), (variant, lam)
    zo = oracle.primal_h16(b, ph, lam)
    assert np.array_equal(z.cpu().numpy().view(np.uint32), zo.view(np.uint32)), (variant, lam)


def test_f16_march_misaligned_falls_back(T):
    """A dual whose base is 8- but not 16-byte aligned cannot feed the
    tensor maps: the fused kernel runs, with the same bits."""
    import torch
    shape = (32, 8, 8)
    n = 32 * 8 * 8
    b = synth.random_case(shape, 51)
    p0 = oracle.float_to_half(synth.random_dual(shape, 52, scale=0.5))
    r0 = oracle.float_to_half(synth.random_dual(shape, 53, scale=0.7))
    ph, rh = p0.copy(), r0.copy()
    oracle.fgp_run_h16(b, ph, rh, 0.05, 3, 1.0)
    pbuf = torch.zeros(3 * n + 4, dtype=torch.float16, device="cuda")
    rbuf = torch.zeros(3 * n + 4, dtype=torch.float16, device="cuda")
    p, r = pbuf[4:], rbuf[4:]                       # 8 bytes past a 256-byte boundary
    p.copy_(dev16(p0).reshape(-1))
    r.copy_(dev16(r0).reshape(-1))
    with T.Tvfgp(*shape) as h:
        h.run_f16(dev(b), p, r, 0.05, 3, 1.0)
        assert h.last_variant == T.TVFGP_VARIANT_FUSED
        assert h.check() == 0
    assert np.array_equal(bits(p).reshape(ph.shape), ph) and np.array_equal(bits(r).reshape(rh.shape), rh)


@pytest.mark.slow
def test_f16_512_cubed_exact(T):
    """The 512^3 workload with a binary16 dual, in the configuration the
    bench times for it (graph replay of the z-march, a fresh b and t0 per
    outer), against the oracle; the first 3 of its 20 outers, to bound the
    oracle's time."""
    w = synth.WORKLOADS["c4"]
    base = synth.phantom(w)
    shape = (3, w.nz, w.ny, w.nx)
    ph = np.zeros(shape, np.uint16)
    rh = np.zeros(shape, np.uint16)
    p, r = dev16(ph), dev16(rh)
    with T.Tvfgp(w.nx, w.ny, w.nz, "auto", True) as h:
        for k in range(3):
            b = synth.make_b(w, k, base)
            h.run_f16(dev(b), p, r, w.lam, w.steps, w.t0)
            oracle.fgp_run_h16(b, ph, rh, w.lam, w.steps, w.t0)
        assert h.last_variant == T.TVFGP_VARIANT_ZMARCH_TMA
        assert h.check() == 0
    assert np.array_equal(bits(p), ph) and np.array_equal(bits(r), rh)


def test_accuracy_against_fp32(T):
    """128^3, 50 steps: the denoised volume within 1e-3 max|b| of the fp32
    result (measured 2.6e-4 with the oracles)."""
    import torch
    w = synth.WORKLOADS["c2"]
    b = synth.make_b(w, 0)
    bd = dev(b)
    shape = (3, w.nz, w.ny, w.nx)
    p16 = torch.zeros(shape, dtype=torch.float16, device="cuda")
    r16 = torch.zeros_like(p16)
    p32 = torch.zeros(shape, device="cuda")
    r32 = torch.zeros_like(p32)
    with T.Tvfgp(w.nx, w.ny, w.nz) as h:
        h.run_f16(bd, p16, r16, w.lam, w.steps, 1.0)
        z16 = h.primal_f16(bd, p16, w.lam)
        h.run(bd, p32, r32, w.lam, w.steps, 1.0)
        z32 = h.primal(bd, p32, w.lam)
        h.check()
    assert float((z16 - z32).abs().max()) <= 1e-3 * float(np.abs(b).max())


def test_f16_argument_errors(T):
    import ctypes
    import torch
    n = 8 * 4 * 4
    b = torch.rand(n, device="cuda")
    p = torch.zeros(3 * n + 1, dtype=torch.float16, device="cuda")
    h = T.tvfgp_create(8, 4, 4)
    try:
        tf = ctypes.c_double()
        P = p.data_ptr()
        rb = torch.zeros(3 * n, dtype=torch.float16, device="cuda")
        assert T.raw_call("tvfgp_run_f16", h, b.data_ptr(), P + 1, rb.data_ptr(), 0.1, 2, 1.0, None,
                          ctypes.byref(tf)) == T.TVFGP_ERR_ALIGN
        assert T.raw_call("tvfgp_run_f16", h, b.data_ptr(), P, P, 0.1, 2, 1.0, None,
                          ctypes.byref(tf)) == T.TVFGP_ERR_ARG
        assert T.raw_call("tvfgp_run_f16", h, b.data_ptr(), None, rb.data_ptr(), 0.1, 2, 1.0, None,
                          ctypes.byref(tf)) == T.TVFGP_ERR_ARG
        assert T.tvfgp_launch_count(h) == 0
    finally:
        T.tvfgp_destroy(h)


@pytest.mark.slow
def test_f16_1000x600x300_exact(T):
    """The 1000x600x300 blob volume with a binary16 dual (nx % 8 == 0: the
    z-march), its first 30 steps, against the binary16 oracle."""
    w = synth.WORKLOADS["c5"]
    b = synth.make_b(w, 0, synth.phantom(w))
    shape = (3, w.nz, w.ny, w.nx)
    ph = np.zeros(shape, np.uint16)
    rh = np.zeros(shape, np.uint16)
    p, r = dev16(ph), dev16(rh)
    with T.Tvfgp(w.nx, w.ny, w.nz, "auto", True) as h:
        h.run_f16(dev(b), p, r, w.lam, 30, w.t0)
        assert h.last_variant == T.TVFGP_VARIANT_ZMARCH_TMA
        assert h.check() == 0
    oracle.fgp_run_h16(b, ph, rh, w.lam, 30, w.t0)
    assert np.array_equal(bits(p), ph) and np.array_equal(bits(r), rh)


def random_f16_shapes(count, seed):
    rng = np.random.default_rng(seed)
    out = []
    for k in range(count):
        nx = int(rng.integers(1, 25)) * 8 if k % 3 else int(rng.integers(1, 120))
        out.append((nx, int(rng.integers(1, 70)), int(rng.integers(1, 100))))
    return out


@pytest.mark.parametrize("shape", random_f16_shapes(8, 20261204))
def test_random_shapes_exact(T, shape):
    nx, ny, nz = shape
    seed = (nx * 131 + ny) * 197 + nz
    rng = np.random.default_rng(seed)
    nsteps = int(rng.integers(1, 10))
    lam = float(rng.uniform(0.01, 0.2))
    b = synth.random_case(shape, seed)
    p0 = oracle.float_to_half(synth.random_dual(shape, seed + 1, scale=0.5))
    r0 = oracle.float_to_half(synth.random_dual(shape, seed + 2, scale=0.7))
    p, r = dev16(p0), dev16(r0)
    with T.Tvfgp(nx, ny, nz) as h:
        h.run_f16(dev(b), p, r, lam, nsteps, 1.0)
        assert h.last_variant == expected_variant(T, nx, "auto")
        assert h.check() == 0
    ph, rh = p0.copy(), r0.copy()
    oracle.fgp_run_h16(b, ph, rh, lam, nsteps, 1.0)
    assert np.array_equal(bits(p), ph), (shape, nsteps, lam)
    assert np.array_equal(bits(r), rh), (shape, nsteps, lam)
