"""Parity at the edges of fp32, through every variant: bit patterns of p, r
and z (so signed zeros count) against the oracle on inputs that drive the
projection off its fast path or into subnormals.

- tiny lambda: s = 1/(12 lambda) is about 8e15, so |q|^2 passes 2^100 and
  the projection takes its IEEE fallback;
- mixed magnitudes: dual components from 1e-30 to 1e10 in one vector, and
  half of b negative so that z clamps to 0 and g vanishes (q = r there):
  tiny components next to large ones;
- subnormal b and dual: every value below the normal range;
- huge lambda: s is about 8e-32, so q is r up to rounding."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

SHAPE = (40, 13, 9)
CASES = ["tiny_lambda", "mixed_magnitudes", "subnormal_b", "huge_lambda"]
VARIANTS = ["auto", "zmarch2", "zmarch", "fused", "scalar", "separate", "cube"]


def make_case(name, seed=5):
    nx, ny, nz = SHAPE
    g = np.random.default_rng(seed)
    vol, dual = (nz, ny, nx), (3, nz, ny, nx)
    if name == "tiny_lambda":
        return (g.uniform(0, 1, vol), g.uniform(-1, 1, dual), g.uniform(-1, 1, dual), 1e-17)
    if name == "mixed_magnitudes":
        vals = np.float32([0, 1e-30, -1e-30, 1e-20, -3e-39, 0.3, -0.3, 1.7, -1.7, 1e10, -1e10])
        b = np.where(g.uniform(size=vol) < 0.5, -1.0, g.uniform(0, 1, vol))
        return b, g.choice(vals, size=dual), g.choice(vals, size=dual), 0.05
    if name == "subnormal_b":
        return (g.uniform(0, 1, vol) * 1e-40, g.uniform(-0.5, 0.5, dual) * 1e-38,
                g.uniform(-0.5, 0.5, dual) * 1e-38, 1e-3)
    if name == "huge_lambda":
        return g.uniform(0, 1e4, vol), g.uniform(-2, 2, dual), g.uniform(-2, 2, dual), 1e30
    raise KeyError(name)


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("variant", VARIANTS)
def test_extreme_inputs_bitwise(case, variant):
    import torch
    from fgp_dual_stencil_gb300 import tvfgp as T
    b, p0, r0, lam = make_case(case)
    b, p0, r0 = (np.ascontiguousarray(a, dtype=np.float32) for a in (b, p0, r0))
    nx, ny, nz = SHAPE
    nsteps = 5
    p, r = torch.from_numpy(p0.copy()).cuda(), torch.from_numpy(r0.copy()).cuda()
    bd = torch.from_numpy(b).cuda()
    with T.Tvfgp(nx, ny, nz, variant) as h:
        h.run(bd, p, r, lam, nsteps, 1.0)
        z = h.primal(bd, p, lam)
        assert h.check() == 0
    po, ro = p0.copy(), r0.copy()
    oracle.fgp_run(b, po, ro, lam, nsteps, 1.0)
    zo = oracle.primal(b, po, lam)
    assert np.isfinite(po).all() and np.isfinite(ro).all() and np.isfinite(zo).all()
    assert np.array_equal(bits(p.cpu().numpy()), bits(po)), (case, variant, "p")
    assert np.array_equal(bits(r.cpu().numpy()), bits(ro)), (case, variant, "r")
    assert np.array_equal(bits(z.cpu().numpy()), bits(zo)), (case, variant, "z")
