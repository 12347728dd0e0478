"""The step kernels project q onto the unit ball with a square-root estimate
and fused multiply-add corrections; the step is defined by the IEEE square
root and division (the oracle uses them), so the fast path must return the
same bits.  These tests run its self-check on the GPU: exhaustively for the
square root and reciprocal, on 2^32 random triples for the whole projection,
on 2^32 quotients, half of them next to a power of two, and on 2^28
random quads through the kernels' four-voxel update."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available()
    from fgp_dual_stencil_gb300 import tvfgp
    return tvfgp


def run_check(T, mode, count, seed):
    import torch
    out = torch.tensor([0, -1], dtype=torch.int64, device="cuda")
    T.tvfgp_debug_projection_check(mode, count, seed, out)
    torch.cuda.synchronize()
    return int(out[0]), int(out[1])


def test_sqrt_and_reciprocal_exhaustive(T):
    bad, first = run_check(T, 0, 0, 0)
    assert bad == 0, "%d values of |q|^2 in [1, 2^100) differ, the first at %#x" % (bad, 0x3f800000 + first)


@pytest.mark.parametrize("seed", [1, 0x5eed])
def test_projection_random_triples(T, seed):
    bad, first = run_check(T, 1, 1 << 32, seed)
    assert bad == 0, "%d of 2^32 triples differ (first sample %d)" % (bad, first)


@pytest.mark.parametrize("seed", [2, 0xd1de])
def test_quotients_near_binade_edges(T, seed):
    bad, first = run_check(T, 2, 1 << 32, seed)
    assert bad == 0, "%d of 2^32 quotients differ (first sample %d)" % (bad, first)


@pytest.mark.parametrize("seed", [3, 0xface])
def test_quad_update_random(T, seed):
    bad, first = run_check(T, 3, 1 << 28, seed)
    assert bad == 0, "%d of 2^28 quads differ (first sample %d)" % (bad, first)


def test_check_argument_errors(T):
    import torch
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    assert T.raw_call("tvfgp_debug_projection_check", 4, 10, 0, out.data_ptr(), None) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_debug_projection_check", 1, (1 << 40) + 1, 0, out.data_ptr(), None) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_debug_projection_check", 1, 10, 0, None, None) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_debug_projection_check", 1, 10, 0, out.data_ptr() + 4, None) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_debug_projection_check", 1, 0, 0, out.data_ptr(), None) == T.TVFGP_OK
