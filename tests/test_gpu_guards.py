"""Guard bands around every caller buffer: each buffer is the middle of a
larger allocation whose margins hold a canary pattern (a quiet NaN with a
payload).  After runs of every kernel on ragged shapes, the canaries must
be intact (no write outside a buffer) and the results must equal the
oracle's."""
import numpy as np
import pytest

import oracle
from fgp_dual_stencil_gb300 import synth
from gpu_util import Guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available()
    from fgp_dual_stencil_gb300 import tvfgp
    return tvfgp


SHAPES = [(5, 3, 7), (36, 13, 9), (68, 27, 21), (132, 9, 11)]


@pytest.mark.parametrize("variant", ["auto", "fused", "zmarch", "zmarch2", "scalar", "separate", "cube"])
@pytest.mark.parametrize("shape", SHAPES)
def test_no_write_outside_the_buffers(T, shape, variant):
    nx, ny, nz = shape
    b = synth.random_case(shape, 101)
    p0 = synth.random_dual(shape, 102, scale=0.4)
    r0 = synth.random_dual(shape, 103, scale=0.6)
    gb, gp, gr = Guarded(b), Guarded(p0), Guarded(r0)
    gz = Guarded(np.zeros_like(b))
    with T.Tvfgp(nx, ny, nz, variant) as h:
        h.run(gb.t, gp.t, gr.t, 0.07, 7, 1.0)
        h.primal(gb.t, gp.t, 0.07, z=gz.t)
        assert h.check() == 0
    for name, g in (("b", gb), ("p", gp), ("r", gr), ("z", gz)):
        assert g.intact(), "%s: a canary was overwritten (%s, %s)" % (name, variant, shape)
    po, ro = p0.copy(), r0.copy()
    oracle.fgp_run(b, po, ro, 0.07, 7, 1.0)
    assert np.array_equal(gp.values().view(np.float32), po.reshape(-1))
    assert np.array_equal(gr.values().view(np.float32), ro.reshape(-1))
    assert np.array_equal(gz.values().view(np.float32), oracle.primal(b, po, 0.07).reshape(-1))


@pytest.mark.parametrize("shape", [(40, 13, 9), (36, 13, 9), (5, 3, 7)])
def test_no_write_outside_the_binary16_buffers(T, shape):
    nx, ny, nz = shape
    b = synth.random_case(shape, 111)
    p0 = oracle.float_to_half(synth.random_dual(shape, 112, scale=0.4))
    r0 = oracle.float_to_half(synth.random_dual(shape, 113, scale=0.6))
    gb, gp, gr = Guarded(b), Guarded(p0, 16), Guarded(r0, 16)
    gz = Guarded(np.zeros_like(b))
    with T.Tvfgp(nx, ny, nz) as h:
        h.run_f16(gb.t, gp.t, gr.t, 0.07, 7, 1.0)
        h.primal_f16(gb.t, gp.t, 0.07, z=gz.t)
        assert h.check() == 0
    for name, g in (("b", gb), ("p", gp), ("r", gr), ("z", gz)):
        assert g.intact(), "%s: a canary was overwritten (%s)" % (name, shape)
    ph, rh = p0.copy(), r0.copy()
    oracle.fgp_run_h16(b, ph, rh, 0.07, 7, 1.0)
    assert np.array_equal(gp.values(), ph.reshape(-1)) and np.array_equal(gr.values(), rh.reshape(-1))
