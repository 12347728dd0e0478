"""Pins of the CPU oracle against what the page and the mathematics fix.

The method is the FGP step of the page "TV solver: the FGP step on the GPU",
section "What one step does".  None of these checks re-types the oracle's own
stencil: they use hand-derived values, closed forms, exact symmetries, a
matrix form built from the definition of the forward difference, and the
duality gap of the TV-denoising problem the step solves.
"""
import numpy as np
import pytest
import scipy.sparse as sp

import oracle
from fgp_dual_stencil_gb300 import synth
import golden_io


# ---------------------------------------------------------------------------
# independent helpers: the forward difference as a sparse matrix, and the
# primal / dual objectives of  min_{x>=0} |x-b|^2 + 2 lam TV(x)
# ---------------------------------------------------------------------------

def diff_matrix(shape, zero_at_face):
    """(3N x N) forward difference (Dx)_a(i) = x(i) - x(i+e_a).  At the upper
    face of axis a the row is all zero (zero_at_face) or keeps only x(i)
    (x extended by zeros above the volume)."""
    nx, ny, nz = shape
    N = nx * ny * nz
    rows, cols, vals = [], [], []
    strides = (1, nx, nx * ny)
    for z in range(nz):
        for y in range(ny):
            for x in range(nx):
                i = x + nx * (y + ny * z)
                coord = (x, y, z)
                for a, n_a in enumerate((nx, ny, nz)):
                    row = a * N + i
                    inside = coord[a] < n_a - 1
                    if inside or not zero_at_face:
                        rows.append(row); cols.append(i); vals.append(1.0)
                    if inside:
                        rows.append(row); cols.append(i + strides[a]); vals.append(-1.0)
    return sp.csr_matrix((vals, (rows, cols)), shape=(3 * N, N))


def primal_objective(x, b, lam, D):
    g = (D @ x.ravel()).reshape(3, -1)
    tv = np.sqrt((g * g).sum(axis=0)).sum()
    return float(((x - b) ** 2).sum() + 2.0 * lam * tv)


def dual_objective(p, b, lam, D):
    w = b.ravel() - lam * (D.T @ p.reshape(-1))
    return float((b * b).sum() + (np.minimum(w, 0.0) ** 2).sum() - (w * w).sum())


def matrix_step(b, p, r, lam, m):
    """One FGP step in matrix form (float64)."""
    nz, ny, nx = b.shape
    shape = (nx, ny, nz)
    Dpad = diff_matrix(shape, zero_at_face=False)
    Dface = diff_matrix(shape, zero_at_face=True)
    z = np.maximum(b.ravel() - lam * (Dpad.T @ r.reshape(-1)), 0.0)
    g = (Dface @ z).reshape(3, -1)
    q = r.reshape(3, -1) + g / (12.0 * lam)
    n = np.sqrt((q * q).sum(axis=0))
    pp = q / np.maximum(1.0, n)
    rn = pp + m * (pp - p.reshape(3, -1))
    return pp.reshape(p.shape), rn.reshape(r.shape), z.reshape(b.shape)


def zeros_dual(b):
    return np.zeros((3,) + b.shape, dtype=b.dtype)


def faces_zero(f):
    return (np.all(f[0][:, :, -1] == 0) and np.all(f[1][:, -1, :] == 0)
            and np.all(f[2][-1, :, :] == 0))


# ---------------------------------------------------------------------------
# momentum schedule
# ---------------------------------------------------------------------------

def test_momentum_schedule_properties():
    K = 200
    m, tK = oracle.momentum(1.0, K)
    ts = [1.0] + [oracle.momentum(1.0, k)[1] for k in range(1, K + 1)]
    assert tK == ts[-1]
    # t_{k+1} is the positive root of t^2 - t - t_k^2 = 0
    for k in range(K):
        t, tn = ts[k], ts[k + 1]
        assert abs(tn * tn - tn - t * t) <= 1e-12 * tn * tn
        assert tn >= (k + 3) / 2.0 - 1e-12          # t_k >= (k+2)/2 from t_0 = 1
        assert m[k] * tn == pytest.approx(t - 1.0, rel=1e-15, abs=1e-300)
    assert m[0] == 0.0                                 # t0 = 1 starts without momentum
    assert ts[1] == pytest.approx((1 + 5 ** 0.5) / 2, rel=1e-15)
    assert np.all(np.diff(m) > 0) and m[-1] < 1.0
    # restarting from the returned t continues the same sequence
    m1, t1 = oracle.momentum(1.0, 50)
    m2, _ = oracle.momentum(t1, 150)
    assert np.array_equal(np.concatenate([m1, m2]), m)
    m0, t0f = oracle.momentum(2.5, 0)
    assert m0.size == 0 and t0f == 2.5


# ---------------------------------------------------------------------------
# hand-derived steps (tests/golden/hand_steps.txt)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,tol", [(np.float32, 2e-7), (np.float64, 1e-15)])
def test_hand_steps(dtype, tol):
    for case in golden_io.hand_steps():
        b = case["b"].astype(dtype)
        p = zeros_dual(b)
        r = zeros_dual(b)
        oracle.fgp_run(b, p, r, case["lam"], case["steps"], 1.0)
        z = oracle.primal(b, p, case["lam"])
        exp = golden_io.expected_fields(case)
        for name, got in (("p", p), ("r", r), ("z", z)):
            err = np.abs(got.astype(np.float64) - exp[name]).max()
            assert err <= tol * 4, (case["name"], name, err)


# ---------------------------------------------------------------------------
# the matrix form built from the definition of the forward difference
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(5, 3, 4), (1, 1, 1), (2, 1, 1), (1, 4, 3), (3, 1, 5), (6, 5, 2)])
def test_step_matches_matrix_form(shape):
    rng = np.random.default_rng(sum(shape) * 7 + shape[0])
    nx, ny, nz = shape
    b = rng.uniform(-0.3, 1.2, size=(nz, ny, nx))
    p = rng.uniform(-0.6, 0.6, size=(3, nz, ny, nx))
    r = rng.uniform(-0.8, 0.8, size=(3, nz, ny, nx))     # upper faces not zero on purpose
    lam, m = 0.07, 0.3
    pp_ref, rn_ref, z_ref = matrix_step(b, p, r, lam, m)

    p64 = p.copy()
    rn64, z64 = oracle.fgp_step(b, p64, r, lam, m)
    assert np.abs(z64 - z_ref).max() <= 1e-13
    assert np.abs(p64 - pp_ref).max() <= 1e-13
    assert np.abs(rn64 - rn_ref).max() <= 1e-13

    b32, p32, r32 = b.astype(np.float32), p.astype(np.float32), r.astype(np.float32)
    pp_ref32, rn_ref32, z_ref32 = matrix_step(b32.astype(np.float64), p32.astype(np.float64),
                                              r32.astype(np.float64), lam, float(np.float32(m)))
    rn32, z32 = oracle.fgp_step(b32, p32, r32, np.float32(lam), np.float32(m))
    assert np.abs(z32 - z_ref32).max() <= 2e-6
    assert np.abs(p32 - pp_ref32).max() <= 2e-6
    assert np.abs(rn32 - rn_ref32).max() <= 2e-6


def test_adjoint_identity():
    rng = np.random.default_rng(3)
    for shape in [(7, 5, 4), (1, 6, 3), (4, 1, 1)]:
        nx, ny, nz = shape
        z = rng.standard_normal((nz, ny, nx))
        r = rng.standard_normal((3, nz, ny, nx))
        # (1) fully random r, z extended by zeros above the volume
        lhs = float((oracle.adjoint(r) * z).sum())
        zp = np.pad(z, ((0, 1), (0, 1), (0, 1)))
        fwd = [z - zp[:nz, :ny, 1:nx + 1], z - zp[:nz, 1:ny + 1, :nx], z - zp[1:nz + 1, :ny, :nx]]
        rhs = float(sum((r[a] * fwd[a]).sum() for a in range(3)))
        assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + np.abs(r).sum())
        # (2) r with zero upper faces against the gradient with g_a = 0 at the face
        r[0][:, :, -1] = 0
        r[1][:, -1, :] = 0
        r[2][-1, :, :] = 0
        lhs = float((oracle.adjoint(r) * z).sum())
        rhs = float((r * oracle.gradient(z)).sum())
        assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + np.abs(r).sum())


# ---------------------------------------------------------------------------
# special cases and invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("c", [0.7, -0.3, 0.0])
def test_constant_b_keeps_dual_zero(c):
    b = np.full((6, 5, 7), c, dtype=np.float32)
    p, r = zeros_dual(b), zeros_dual(b)
    oracle.fgp_run(b, p, r, 0.05, 15, 1.0)
    assert not p.any() and not r.any()
    assert np.array_equal(oracle.primal(b, p, 0.05), np.maximum(b, 0))


def test_invariants_on_ellipsoid_workload():
    w = synth.WORKLOADS["c1"]
    b = synth.make_b(w, 0)
    p, r = zeros_dual(b), zeros_dual(b)
    oracle.fgp_run(b, p, r, w.lam, w.steps, w.t0)
    z = oracle.primal(b, p, w.lam)
    nrm = np.sqrt((p.astype(np.float64) ** 2).sum(axis=0))
    assert nrm.max() <= 1.0 + 2.0 ** -22
    assert nrm.max() > 0.5                      # the projection is exercised
    assert z.min() >= 0.0 and (z == 0).any()    # the clamp is exercised
    assert faces_zero(p) and faces_zero(r)


def test_fp32_against_fp64_drift_within_tolerance():
    """fp32 rounding after the ellipsoid workload stays far inside 1e-5."""
    w = synth.WORKLOADS["c1"]
    b = synth.make_b(w, 0)
    p32, r32 = zeros_dual(b), zeros_dual(b)
    oracle.fgp_run(b, p32, r32, w.lam, w.steps, w.t0)
    b64 = b.astype(np.float64)
    p64, r64 = zeros_dual(b64), zeros_dual(b64)
    oracle.fgp_run(b64, p64, r64, float(np.float32(w.lam)), w.steps, w.t0)
    assert np.abs(p32 - p64).max() < 1e-5
    assert np.abs(r32 - r64).max() < 1e-5


@pytest.mark.parametrize("axis", [0, 1, 2])
@pytest.mark.parametrize("b0,b1,lam", [(0.9, 0.5, 0.05), (0.9, 0.5, 0.4), (0.2, 0.6, 0.1)])
def test_two_voxel_closed_form(axis, b0, b1, lam):
    shape = [1, 1, 1]
    shape[axis] = 2
    nx, ny, nz = shape
    b = np.zeros((nz, ny, nx))
    idx0 = [0, 0, 0]
    idx1 = [0, 0, 0]
    idx1[2 - axis] = 1
    b[tuple(idx0)] = b0
    b[tuple(idx1)] = b1
    pstar = np.clip((b0 - b1) / (2 * lam), -1.0, 1.0)
    zstar = (b0 - lam * pstar, b1 + lam * pstar)
    for dtype, tol in ((np.float64, 1e-6), (np.float32, 1e-5)):
        bb = b.astype(dtype)
        p, r = zeros_dual(bb), zeros_dual(bb)
        oracle.fgp_run(bb, p, r, lam, 2000, 1.0)
        z = oracle.primal(bb, p, lam)
        assert abs(float(p[axis][tuple(idx0)]) - pstar) <= tol
        assert abs(float(z[tuple(idx0)]) - zstar[0]) <= tol
        assert abs(float(z[tuple(idx1)]) - zstar[1]) <= tol
        assert float(p[axis][tuple(idx1)]) == 0.0


@pytest.mark.parametrize("k", [3, -2, 7])
def test_power_of_two_scaling_is_exact(k):
    rng = np.random.default_rng(11)
    b = rng.uniform(-0.2, 1.0, size=(9, 8, 10)).astype(np.float32)
    lam = np.float32(0.04)
    s = np.float32(2.0 ** k)
    p1, r1 = zeros_dual(b), zeros_dual(b)
    oracle.fgp_run(b, p1, r1, lam, 25, 1.0)
    p2, r2 = zeros_dual(b), zeros_dual(b)
    oracle.fgp_run(b * s, p2, r2, lam * s, 25, 1.0)
    assert np.array_equal(p1, p2) and np.array_equal(r1, r2)
    assert np.array_equal(oracle.primal(b, p1, lam) * s, oracle.primal(b * s, p2, lam * s))


def test_transpose_equivariance():
    rng = np.random.default_rng(5)
    b = rng.uniform(-0.2, 1.0, size=(4, 6, 9)).astype(np.float32)    # (nz, ny, nx)
    lam = 0.06
    p, r = zeros_dual(b), zeros_dual(b)
    oracle.fgp_run(b, p, r, lam, 20, 1.0)
    # x <-> y: exact (the two terms that swap are added first, and addition commutes)
    bt = np.ascontiguousarray(b.transpose(0, 2, 1))
    pt, rt = zeros_dual(bt), zeros_dual(bt)
    oracle.fgp_run(bt, pt, rt, lam, 20, 1.0)
    assert np.array_equal(pt[0], p[1].transpose(0, 2, 1))
    assert np.array_equal(pt[1], p[0].transpose(0, 2, 1))
    assert np.array_equal(pt[2], p[2].transpose(0, 2, 1))
    assert np.array_equal(rt[0], r[1].transpose(0, 2, 1))
    # x <-> z: equal up to the order of the sum in L(r)
    bz = np.ascontiguousarray(b.transpose(2, 1, 0))
    pz, rz = zeros_dual(bz), zeros_dual(bz)
    oracle.fgp_run(bz, pz, rz, lam, 20, 1.0)
    assert np.abs(pz[0] - p[2].transpose(2, 1, 0)).max() <= 1e-6
    assert np.abs(pz[2] - p[0].transpose(2, 1, 0)).max() <= 1e-6
    assert np.abs(pz[1] - p[1].transpose(2, 1, 0)).max() <= 1e-6


def test_thread_count_does_not_change_results():
    w = synth.WORKLOADS["c1"]
    b = synth.make_b(w, 0)
    out = []
    n0 = oracle.get_threads()
    try:
        for n in (1, max(2, n0)):
            oracle.set_threads(n)
            p, r = zeros_dual(b), zeros_dual(b)
            oracle.fgp_run(b, p, r, w.lam, w.steps, 1.0)
            out.append((p, r))
    finally:
        oracle.set_threads(n0)
    assert np.array_equal(out[0][0], out[1][0]) and np.array_equal(out[0][1], out[1][1])


# ---------------------------------------------------------------------------
# convergence to the TV prox, certified by the duality gap
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape,lam", [((4, 4, 4), 0.1), ((5, 3, 6), 0.05)])
def test_fgp_converges_to_certified_tv_prox(shape, lam):
    nx, ny, nz = shape
    rng = np.random.default_rng(nx * 100 + nz)
    b = np.zeros((nz, ny, nx))
    b[: nz // 2 + 1, :, : nx // 2] = 0.8
    b += rng.uniform(0.0, 0.3, size=b.shape)
    Dface = diff_matrix(shape, zero_at_face=True)

    p, r = zeros_dual(b), zeros_dual(b)
    gaps = []
    t = 1.0
    for chunk in (100, 900, 4000, 15000):
        t = oracle.fgp_run(b, p, r, lam, chunk, t)
        x = oracle.primal(b, p, lam)
        assert faces_zero(p)
        assert np.sqrt((p ** 2).sum(axis=0)).max() <= 1.0 + 1e-12
        gap = primal_objective(x, b, lam, Dface) - dual_objective(p, b, lam, Dface)
        assert gap >= -1e-12                       # weak duality
        gaps.append(gap)
    assert gaps[0] > gaps[1] > gaps[-1]
    # 2-strong convexity: |x - x*|^2 <= gap, so x is within sqrt(gap) of the prox
    assert gaps[-1] <= 1e-11 * (1.0 + (b * b).sum())
    x_star = x

    b32 = b.astype(np.float32)
    p32, r32 = zeros_dual(b32), zeros_dual(b32)
    oracle.fgp_run(b32, p32, r32, lam, 5000, 1.0)
    z32 = oracle.primal(b32, p32, lam)
    assert np.abs(z32 - x_star).max() <= 1e-4


def tv1d_brute_force(y, lam):
    """Exact minimiser of 1/2 |x - y|^2 + lam * sum_i |x(i+1) - x(i)| for a
    short signal, by enumeration.  With u the dual (x = y - D^T u, where
    (D^T u)(i) = u(i-1) - u(i) and u(-1) = u(n-1) = 0), optimality makes x
    constant on runs between jumps and u = lam * sign(jump) at each jump, so
    summing x = y - D^T u over a run [a, e] gives its value
    mean(y[a..e]) - (u(a-1) - u(e)) / (e - a + 1).  Every choice, per edge,
    of "no jump", "up" or "down" yields such a candidate; the optimum is one
    of them, and since each candidate is a feasible point, it is the one of
    least objective."""
    import itertools
    n = len(y)
    best, best_x = np.inf, None
    for pattern in itertools.product((0, 1, -1), repeat=n - 1):
        x = np.empty(n)
        a = 0
        for e in range(n):
            if e == n - 1 or pattern[e] != 0:
                u_left = lam * pattern[a - 1] if a > 0 else 0.0
                u_right = lam * pattern[e] if e < n - 1 else 0.0
                x[a:e + 1] = y[a:e + 1].mean() - (u_left - u_right) / (e - a + 1)
                a = e + 1
        obj = 0.5 * ((x - y) ** 2).sum() + lam * np.abs(np.diff(x)).sum()
        if obj < best:
            best, best_x = obj, x
    return best_x


def test_tv1d_brute_force_on_hand_cases():
    # no jump can pay for itself when lam is large: the mean
    y = np.array([0.1, 0.9, 0.3, 0.7])
    assert np.allclose(tv1d_brute_force(y, 10.0), y.mean())
    # a single step: each run moves towards the other by lam / (its length)
    y = np.array([0.0, 0.0, 1.0, 1.0])
    assert np.allclose(tv1d_brute_force(y, 0.1), [0.05, 0.05, 0.95, 0.95])
    # lam -> 0 gives y back
    y = np.array([0.3, 0.1, 0.4, 0.1, 0.5])
    assert np.allclose(tv1d_brute_force(y, 1e-9), y, atol=1e-8)


@pytest.mark.parametrize("axis", [0, 1, 2])
@pytest.mark.parametrize("n,lam,seed", [(7, 0.05, 1), (8, 0.1, 2), (9, 0.02, 3)])
def test_fgp_on_a_line_is_1d_tv_denoising(axis, n, lam, seed):
    """On an n x 1 x 1 volume (or its y / z twins) with b >= 0 the prox is
    plain 1D TV denoising (x >= 0 is inactive by the maximum principle), so a
    long FGP run must reach the brute-force minimiser."""
    rng = np.random.default_rng(seed)
    y = np.clip(np.repeat(rng.uniform(0.0, 1.0, size=3), [2, n - 4, 2]) + rng.normal(0.0, 0.1, size=n), 0.0, None)
    x_star = tv1d_brute_force(y, lam)
    shape = [1, 1, 1]
    shape[2 - axis] = n                        # arrays are (nz, ny, nx)
    b = y.reshape(shape)
    p, r = zeros_dual(b), zeros_dual(b)
    oracle.fgp_run(b, p, r, lam, 20000, 1.0)
    z = oracle.primal(b, p, lam).ravel()
    assert np.abs(z - x_star).max() <= 1e-6
    # the other components of the dual stay exactly 0
    for a in range(3):
        if a != axis:
            assert np.all(p[a] == 0) and np.all(r[a] == 0)
    b32 = b.astype(np.float32)
    p32, r32 = zeros_dual(b32), zeros_dual(b32)
    oracle.fgp_run(b32, p32, r32, lam, 5000, 1.0)
    assert np.abs(oracle.primal(b32, p32, lam).ravel() - x_star).max() <= 1e-4


# ---------------------------------------------------------------------------
# binary16 storage of the dual
# ---------------------------------------------------------------------------

def test_half_conversions_match_ieee_binary16():
    h = np.arange(65536, dtype=np.uint16)
    f = oracle.half_to_float(h)
    ref = h.view(np.float16).astype(np.float32)            # numpy's IEEE binary16
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(f), nan)
    assert np.array_equal(f[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(400_000) * np.exp(rng.uniform(-20, 12, 400_000))).astype(np.float32)
    # exact halfway cases between neighbouring binary16 values: ties to even
    finite = np.isfinite(ref[:-1]) & np.isfinite(ref[1:])
    mids = (ref[:-1][finite].astype(np.float64) + ref[1:][finite].astype(np.float64)) / 2
    mids = mids[np.abs(mids) < 65504].astype(np.float32)
    x = np.concatenate([x, mids, np.array([0.0, -0.0, 65504, 65519.9, 65520, 1e-8, -6e-8], np.float32)])
    with np.errstate(over="ignore"):
        assert np.array_equal(oracle.float_to_half(x), x.astype(np.float16).view(np.uint16))


def test_half_storage_step_is_the_fp32_step_rounded():
    """One step with binary16 storage equals the matrix-form step on the
    widened inputs, rounded to binary16 by numpy."""
    shape = (6, 5, 4)
    nx, ny, nz = shape
    rng = np.random.default_rng(21)
    b = rng.uniform(-0.2, 1.2, size=(nz, ny, nx)).astype(np.float32)
    p16 = rng.uniform(-0.6, 0.6, size=(3, nz, ny, nx)).astype(np.float16)
    r16 = rng.uniform(-0.8, 0.8, size=(3, nz, ny, nx)).astype(np.float16)
    lam, m = np.float32(0.07), np.float32(0.3)
    p32, r32 = p16.astype(np.float32), r16.astype(np.float32)
    rd32, _ = oracle.fgp_step(b, p32, r32, lam, m)                  # fp32 step on widened values
    ph = p16.view(np.uint16).copy()
    rdh = oracle.fgp_step_h16(b, ph, r16.view(np.uint16).copy(), lam, m)
    assert np.array_equal(ph, p32.astype(np.float16).view(np.uint16))
    assert np.array_equal(rdh, rd32.astype(np.float16).view(np.uint16))
    # and the fp32 step itself agrees with the matrix form
    pp_ref, rn_ref, _ = matrix_step(b.astype(np.float64), p16.astype(np.float64), r16.astype(np.float64),
                                    float(lam), float(m))
    assert np.abs(p32 - pp_ref).max() <= 2e-6 and np.abs(rd32 - rn_ref).max() <= 2e-6


def test_half_storage_changes_the_result_only_slightly():
    """Measured drift of the half-storage dual on the 32^3 workload: the
    denoised volume stays within 1e-3 max|b| of the fp32 result."""
    w = synth.WORKLOADS["c1"]
    b = synth.make_b(w, 0)
    p, r = zeros_dual(b), zeros_dual(b)
    oracle.fgp_run(b, p, r, w.lam, w.steps, 1.0)
    ph = np.zeros((3,) + b.shape, np.uint16)
    rh = np.zeros_like(ph)
    oracle.fgp_run_h16(b, ph, rh, w.lam, w.steps, 1.0)
    dz = np.abs(oracle.primal_h16(b, ph, w.lam) - oracle.primal(b, p, w.lam)).max()
    assert 0 < dz <= 1e-3 * np.abs(b).max()
    assert np.abs(oracle.half_to_float(ph) - p).max() <= 1e-2
