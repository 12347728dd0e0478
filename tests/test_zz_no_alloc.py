"""tvfgp_run_noalloc, called through the C ABI.

This entry point serves callers that must not allocate device memory (a host
framework that owns the whole memory pool, a plug-in handed only buffers, a
loop that cannot afford the synchronisation of a cudaMalloc).  It keeps its
second r buffer in a fixed array compiled into the library, so these tests
check that it gives the same results as tvfgp_run (which allocates its
scratch in a handle), over two calls in a row, that a volume above the fixed
capacity is refused, and that repeated calls leave the free device memory
unchanged.  The file is named to be collected last."""
import ctypes

import numpy as np
import pytest

from fgp_dual_stencil_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 1e-5                 # the tolerance of the other parity tests on p and r
MAX_VOXELS = 2097152       # TVFGP_NOALLOC_MAX_VOXELS in include/tvfgp.h


def c_entry():
    from fgp_dual_stencil_gb300 import tvfgp as T
    lib = ctypes.CDLL(T.LIB_PATH)
    fn = lib.tvfgp_run_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [i, i, i, vp, vp, vp, ctypes.c_float, i, ctypes.c_double, vp,
                   ctypes.POINTER(ctypes.c_double)]
    fn.restype = i
    return T, fn


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("shape", [(64, 48, 40), (30, 20, 10), (128, 128, 128)])
def test_noalloc_matches_run_over_two_calls(shape):
    import torch
    T, fn = c_entry()
    nx, ny, nz = shape
    lam = 0.04
    b = synth.random_case(shape, 21)
    p0 = synth.random_dual(shape, 22, scale=0.3)
    r0 = synth.random_dual(shape, 23, scale=0.5)
    bd = dev(b)

    # existing entry point (scratch allocated by the handle)
    p_ref, r_ref = dev(p0), dev(r0)
    with T.Tvfgp(nx, ny, nz) as h:
        t_ref = h.run(bd, p_ref, r_ref, lam, 7, 1.0)
        t_ref = h.run(bd, p_ref, r_ref, lam, 4, t_ref)
        assert h.check() == T.TVFGP_OK

    # the entry point that allocates nothing: two calls in a row
    p, r = dev(p0), dev(r0)
    stream = torch.cuda.current_stream().cuda_stream
    tf = ctypes.c_double(0.0)
    assert fn(nx, ny, nz, bd.data_ptr(), p.data_ptr(), r.data_ptr(), lam, 7, 1.0, stream,
              ctypes.byref(tf)) == T.TVFGP_OK
    t1 = tf.value
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    assert fn(nx, ny, nz, bd.data_ptr(), p.data_ptr(), r.data_ptr(), lam, 4, t1, stream,
              ctypes.byref(tf)) == T.TVFGP_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before

    assert tf.value == t_ref
    dp = float((p - p_ref).abs().max())
    dr = float((r - r_ref).abs().max())
    assert dp <= TOL and dr <= TOL, (dp, dr)


def test_noalloc_refuses_volumes_above_its_capacity():
    T, fn = c_entry()
    tf = ctypes.c_double(0.0)
    assert 129 * 128 * 128 > MAX_VOXELS
    rc = fn(129, 128, 128, None, None, None, 0.04, 3, 1.0, None, ctypes.byref(tf))
    assert rc == T.TVFGP_ERR_UNSUPPORTED
    rc = fn(0, 4, 4, None, None, None, 0.04, 3, 1.0, None, ctypes.byref(tf))
    assert rc == T.TVFGP_ERR_ARG
