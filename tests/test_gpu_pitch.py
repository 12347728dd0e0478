"""Volumes with padded rows (tvfgp_create_pitched), such as the in-place
real-to-complex FFT layout with rows of 2*(nx/2+1) floats.  The padding is
filled with garbage; on x < nx the results must equal the oracle's on the
dense volume bit for bit, and the padding must come back untouched."""
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


def pad(a, pitch, seed):
    """a (..., nx) -> (..., pitch) with pseudo-random values in x >= nx."""
    out = np.random.default_rng(seed).uniform(-7, 7, a.shape[:-1] + (pitch,)).astype(a.dtype)
    out[..., :a.shape[-1]] = a
    return out


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pitched_variant(T, nx, pitch, variant="auto", nsteps=1):
    """What a pitched handle runs.  Runs of 4 or more steps with nx % 4 == 0
    on AUTO and the TMA variants go through dense buffers and are reported as
    the dense kernel (on AUTO and ZMARCH2_TMA with an even pitch the first
    step packs and the last launch unpacks); otherwise the fused kernel on 8-byte halves or pairs
    (reported as FUSED) when nx and the pitch are even, else the scalar
    kernel; SCALAR and SEPARATE handles keep theirs."""
    if nsteps >= 4 and nx % 4 == 0 and variant in ("auto", "zmarch", "zmarch2", "cube"):
        return {"auto": T.TVFGP_VARIANT_ZMARCH2_TMA, "zmarch": T.TVFGP_VARIANT_ZMARCH_TMA,
                "zmarch2": T.TVFGP_VARIANT_ZMARCH2_TMA, "cube": T.TVFGP_VARIANT_CUBE_TMA}[variant]
    if variant == "separate":
        return T.TVFGP_VARIANT_SEPARATE
    if variant == "scalar" or nx % 2 or pitch % 2:
        return T.TVFGP_VARIANT_SCALAR
    return T.TVFGP_VARIANT_FUSED


def check(got, want, padded_before, nx, what):
    g = got.detach().cpu().numpy()
    assert np.array_equal(g[..., :nx], want), "%s differs from the oracle" % what
    assert np.array_equal(g[..., nx:], padded_before[..., nx:]), "%s: padding was written" % what


CASES = [((32, 8, 6), None), ((33, 5, 7), None), ((64, 17, 9), None), ((130, 9, 11), None),
         ((7, 3, 2), None), ((40, 6, 5), 45), ((1, 1, 1), 2)]


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("shape,pitch", CASES)
def test_pitched_equals_dense_oracle(T, shape, pitch, graph):
    nx, ny, nz = shape
    pitch = pitch or T.fft_pitch(nx)
    b = synth.random_case(shape, 61)
    p0 = synth.random_dual(shape, 62, scale=0.4)
    r0 = synth.random_dual(shape, 63, scale=0.6)
    bp, pp, rp = pad(b, pitch, 1), pad(p0, pitch, 2), pad(r0, pitch, 3)
    zp = pad(np.zeros_like(b), pitch, 4)
    # 4 and 6: packing step, one dense step, two-step launches; 5: packing
    # step and two-step launches only
    for nsteps in (0, 1, 2, 4, 5, 6):
        p, r, z = dev(pp), dev(rp), dev(zp)
        with T.Tvfgp(nx, ny, nz, "auto", graph, pitch=pitch) as h:
            h.run(dev(bp), p, r, 0.07, nsteps, 1.0)
            h.primal(dev(bp), p, 0.07, z=z)
            assert h.last_variant == pitched_variant(T, nx, pitch, "auto", nsteps) or nsteps == 0
            assert h.check() == 0
        po, ro = p0.copy(), r0.copy()
        oracle.fgp_run(b, po, ro, 0.07, nsteps, 1.0)
        check(p, po, pp, nx, "p")
        check(r, ro, rp, nx, "r")
        check(z, oracle.primal(b, po, 0.07), zp, nx, "z")


@pytest.mark.parametrize("variant", ["separate", "zmarch2", "zmarch", "fused", "scalar", "cube"])
def test_pitched_any_variant(T, variant):
    """Every variant set on a pitched handle runs the float2 fused kernel or a
    scalar kernel (the two-kernel variant its scalar pair), with the same
    bits."""
    shape = (48, 11, 9)
    nx, ny, nz = shape
    pitch = T.fft_pitch(nx)
    b = synth.random_case(shape, 71)
    p0 = synth.random_dual(shape, 72, scale=0.4)
    r0 = synth.random_dual(shape, 73, scale=0.6)
    bp, pp, rp = pad(b, pitch, 5), pad(p0, pitch, 6), pad(r0, pitch, 7)
    p, r = dev(pp), dev(rp)
    with T.Tvfgp(nx, ny, nz, variant, False, pitch=pitch) as h:
        h.run(dev(bp), p, r, 0.05, 6, 1.0)
        assert h.last_variant == pitched_variant(T, nx, pitch, variant, 6)
        assert h.check() == 0
    oracle.fgp_run(b, p0, r0, 0.05, 6, 1.0)
    check(p, p0, pp, nx, "p")
    check(r, r0, rp, nx, "r")


def test_pitched_binary16(T):
    import torch
    shape = (62, 7, 5)
    nx, ny, nz = shape
    pitch = T.fft_pitch(nx)
    b = synth.random_case(shape, 81)
    p0 = oracle.float_to_half(synth.random_dual(shape, 82, scale=0.4))
    r0 = oracle.float_to_half(synth.random_dual(shape, 83, scale=0.6))
    bp = pad(b, pitch, 8)
    pp = pad(p0.view(np.float16), pitch, 9)
    rp = pad(r0.view(np.float16), pitch, 10)
    p, r = dev(pp), dev(rp)
    z = torch.zeros((nz, ny, pitch), device="cuda")
    with T.Tvfgp(nx, ny, nz, pitch=pitch) as h:
        h.run_f16(dev(bp), p, r, 0.05, 5, 1.0)
        h.primal_f16(dev(bp), p, 0.05, z=z)
        assert h.last_variant == T.TVFGP_VARIANT_SCALAR
        assert h.check() == 0
    ph, rh = p0.copy(), r0.copy()
    oracle.fgp_run_h16(b, ph, rh, 0.05, 5, 1.0)
    check(p, ph.view(np.float16), pp, nx, "p (binary16)")
    check(r, rh.view(np.float16), rp, nx, "r (binary16)")
    assert np.array_equal(z.cpu().numpy()[..., :nx], oracle.primal_h16(b, ph, 0.05))


def test_pitched_workload_128(T):
    """The 128^3 workload (50 steps) in the FFT layout, pitch 130."""
    w = synth.WORKLOADS["c2"]
    b = synth.make_b(w, 0)
    pitch = T.fft_pitch(w.nx)
    shape = (3, w.nz, w.ny, w.nx)
    bp = pad(b, pitch, 11)
    pp = pad(np.zeros(shape, np.float32), pitch, 12)
    rp = pad(np.zeros(shape, np.float32), pitch, 13)
    p, r = dev(pp), dev(rp)
    with T.Tvfgp(w.nx, w.ny, w.nz, "auto", True, pitch=pitch) as h:
        h.run(dev(bp), p, r, w.lam, w.steps, w.t0)
        assert h.check() == 0
    po = np.zeros(shape, np.float32)
    ro = np.zeros_like(po)
    oracle.fgp_run(b, po, ro, w.lam, w.steps, w.t0)
    check(p, po, pp, w.nx, "p")
    check(r, ro, rp, w.nx, "r")


@pytest.mark.slow
def test_pitched_512_cubed(T):
    """512^3 with rows of 514 floats (the bench's --pitch fft configuration),
    the first 2 of the workload's 20 outers, against the dense oracle."""
    w = synth.WORKLOADS["c4"]
    base = synth.phantom(w)
    pitch = T.fft_pitch(w.nx)
    shape = (3, w.nz, w.ny, w.nx)
    po = np.zeros(shape, np.float32)
    ro = np.zeros_like(po)
    import torch
    p = torch.zeros((3, w.nz, w.ny, pitch), device="cuda")
    r = torch.zeros_like(p)
    with T.Tvfgp(w.nx, w.ny, w.nz, "auto", True, pitch=pitch) as h:
        for k in range(2):
            b = synth.make_b(w, k, base)
            h.run(dev(pad(b, pitch, 20 + k)), p, r, w.lam, w.steps, w.t0)
            oracle.fgp_run(b, po, ro, w.lam, w.steps, w.t0)
        assert h.check() == 0
    assert np.array_equal(p.cpu().numpy()[..., :w.nx], po)
    assert np.array_equal(r.cpu().numpy()[..., :w.nx], ro)
    assert not p[..., w.nx:].any() and not r[..., w.nx:].any()


def test_pitch_argument_errors(T):
    import ctypes
    h = ctypes.c_void_p()
    assert T.raw_call("tvfgp_create_pitched", 8, 4, 4, 7, ctypes.byref(h)) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_create_pitched", 8, 4, 4, 65536, ctypes.byref(h)) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_create_pitched", 8, 4, 4, 10, None) == T.TVFGP_ERR_ARG


@pytest.mark.slow
def test_pitched_1000x600x300(T):
    """The 1000x600x300 workload (100 steps) with rows of 1002 floats, which
    bench --pitch fft times on the packed path, against the dense oracle."""
    import torch
    from gpu_util import run_workload_oracle
    w = synth.WORKLOADS["c5"]
    b = synth.make_b(w, 0, synth.phantom(w))
    pitch = T.fft_pitch(w.nx)
    p = torch.zeros((3, w.nz, w.ny, pitch), device="cuda")
    r = torch.zeros_like(p)
    with T.Tvfgp(w.nx, w.ny, w.nz, "auto", True, pitch=pitch) as h:
        h.run(dev(pad(b, pitch, 30)), p, r, w.lam, w.steps, w.t0)
        assert h.last_variant == T.TVFGP_VARIANT_ZMARCH2_TMA
        assert h.check() == 0
    _, po, ro, _, _ = run_workload_oracle(w)
    assert np.array_equal(p.cpu().numpy()[..., :w.nx], po)
    assert np.array_equal(r.cpu().numpy()[..., :w.nx], ro)
    assert not p[..., w.nx:].any() and not r[..., w.nx:].any()


@pytest.mark.parametrize("shape,pitch", [((32, 9, 7), None), ((34, 9, 7), None), ((33, 5, 4), None),
                                         ((40, 6, 5), 45)])
def test_pitched_single_step(T, shape, pitch):
    """tvfgp_step on padded rows (the in-place kernels: quads as two halves,
    pairs, or scalar) against one oracle step; r_dst's padding untouched."""
    nx, ny, nz = shape
    pitch = pitch or T.fft_pitch(nx)
    b = synth.random_case(shape, 91)
    p0 = synth.random_dual(shape, 92, scale=0.4)
    r0 = synth.random_dual(shape, 93, scale=0.6)
    bp, pp, rp, rdp = pad(b, pitch, 14), pad(p0, pitch, 15), pad(r0, pitch, 16), pad(np.zeros_like(r0), pitch, 17)
    p, rs, rd = dev(pp), dev(rp), dev(rdp)
    with T.Tvfgp(nx, ny, nz, pitch=pitch) as h:
        h.step(dev(bp), p, rs, rd, 0.06, 0.3)
        assert h.last_variant == pitched_variant(T, nx, pitch)
        assert h.check() == 0
    po = p0.copy()
    ro, _ = oracle.fgp_step(b, po, r0, 0.06, 0.3)
    check(p, po, pp, nx, "p")
    check(rd, ro, rdp, nx, "r_dst")
    check(rs, r0, rp, nx, "r_src")


def random_pitched_cases(count, seed):
    """Shapes and pitches drawn at random: the FFT pitch 2*(nx/2+1) in most
    cases, an arbitrary larger pitch in the rest."""
    rng = np.random.default_rng(seed)
    out = []
    for k in range(count):
        nx = int(rng.integers(1, 40)) * 4 if k % 3 else int(rng.integers(1, 150))
        shape = (nx, int(rng.integers(1, 60)), int(rng.integers(1, 90)))
        pitch = 2 * (nx // 2 + 1) if k % 4 else nx + int(rng.integers(1, 9))
        out.append((shape, pitch))
    return out


@pytest.mark.parametrize("shape,pitch", random_pitched_cases(8, 20261203))
def test_random_pitched_shapes(T, shape, pitch):
    nx, ny, nz = shape
    seed = (nx * 131 + ny) * 197 + nz + pitch
    rng = np.random.default_rng(seed)
    nsteps = int(rng.integers(1, 10))
    lam = float(rng.uniform(0.01, 0.2))
    b = synth.random_case(shape, seed)
    p0 = synth.random_dual(shape, seed + 1, scale=0.5)
    r0 = synth.random_dual(shape, seed + 2, scale=0.7)
    bp, pp, rp = pad(b, pitch, seed + 3), pad(p0, pitch, seed + 4), pad(r0, pitch, seed + 5)
    zp = pad(np.zeros_like(b), pitch, seed + 6)
    p, r, z = dev(pp), dev(rp), dev(zp)
    with T.Tvfgp(nx, ny, nz, "auto", True, pitch=pitch) as h:
        h.run(dev(bp), p, r, lam, nsteps, 1.0)
        h.primal(dev(bp), p, lam, z=z)
        assert h.last_variant == pitched_variant(T, nx, pitch, "auto", nsteps)
        assert h.check() == 0
    po, ro = p0.copy(), r0.copy()
    oracle.fgp_run(b, po, ro, lam, nsteps, 1.0)
    check(p, po, pp, nx, "p")
    check(r, ro, rp, nx, "r")
    check(z, oracle.primal(b, po, lam), zp, nx, "z")
