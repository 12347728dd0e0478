"""Calls recorded into the caller's CUDA graph (torch.cuda.graph): a run on
a capturing stream puts its launches into the captured graph one by one
(the handle's own graph is not replayed inside it) and allocates nothing (a
padded-row handle whose dense buffers do not exist yet runs in place), and
every replay gives the oracle's bits."""
import numpy as np
import pytest

import oracle
from fgp_dual_stencil_gb300 import synth

pytestmark = pytest.mark.gpu

SHAPE = (64, 26, 20)
LAM = 0.05
NSTEPS = 6


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("pitch", [None, 66])
def test_run_and_primal_captured_into_a_cuda_graph(graph, pitch):
    import torch
    from fgp_dual_stencil_gb300 import tvfgp as T
    nx, ny, nz = SHAPE
    px = pitch or nx
    b = synth.random_case(SHAPE, 91)
    p0 = synth.random_dual(SHAPE, 92, scale=0.4)
    r0 = synth.random_dual(SHAPE, 93, scale=0.6)

    def padded(a):
        return torch.from_numpy(np.pad(a, [(0, 0)] * (a.ndim - 1) + [(0, px - nx)])).cuda()

    bd, p, r = padded(b), padded(p0), padded(r0)
    z = torch.zeros_like(bd)
    p_init, r_init = p.clone(), r.clone()
    po, ro = p0.copy(), r0.copy()
    oracle.fgp_run(b, po, ro, LAM, NSTEPS, 1.0)
    zo = oracle.primal(b, po, LAM)
    with T.Tvfgp(nx, ny, nz, "auto", graph, pitch=pitch) as h:
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            h.run(bd, p, r, LAM, NSTEPS, 1.0)
            h.primal(bd, p, LAM, z=z)
        torch.cuda.synchronize()
        assert torch.equal(p, p_init) and torch.equal(r, r_init)   # captured, not run
        for _ in range(2):
            p.copy_(p_init)
            r.copy_(r_init)
            z.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(p.cpu().numpy()[..., :nx], po)
            assert np.array_equal(r.cpu().numpy()[..., :nx], ro)
            assert np.array_equal(z.cpu().numpy()[..., :nx], zo)
        assert h.check() == 0
        del g
