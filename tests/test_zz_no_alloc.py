"""tvfgp_run_noalloc, called through the C ABI.

This entry point serves callers that must not allocate device memory: a host
framework that owns the whole device memory pool and hands the library only
buffers, a plug-in that is given fixed buffers, or a loop that cannot afford
the device-wide synchronisation a cudaMalloc or cudaFree may cause.  It keeps
its second r buffer in a fixed array compiled into the library.

These tests check, over two calls in a row, that its results equal the CPU
oracle's and tvfgp_run's bit for bit and that the calls leave the free device
memory unchanged; that a volume above the fixed capacity is refused; that
buffers overlapping the built-in array are refused before anything runs;
that it writes nothing outside the caller's buffers (guard bands); and that
a first call in a process made under stream capture is refused.  The file is
named to be collected last."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from fgp_dual_stencil_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 1e-5                 # the bar of the parity tests on p and r (the tests demand equality)
MAX_VOXELS = 2097152       # TVFGP_NOALLOC_MAX_VOXELS in include/tvfgp.h
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
def test_noalloc_matches_oracle_and_run_over_two_calls(shape):
    import torch
    T, fn = c_entry()
    nx, ny, nz = shape
    lam = 0.04
    b = synth.random_case(shape, 21)
    p0 = synth.random_dual(shape, 22, scale=0.3)
    r0 = synth.random_dual(shape, 23, scale=0.5)
    bd = dev(b)
    stream = torch.cuda.current_stream().cuda_stream

    # the oracle: 7 steps from t0 = 1, then 4 more from the t it returned
    po, ro = p0.copy(), r0.copy()
    t1o = oracle.fgp_run(b, po, ro, lam, 7, 1.0)
    t2o = oracle.fgp_run(b, po, ro, lam, 4, t1o)

    # the existing entry point (scratch allocated by the handle)
    p_ref, r_ref = dev(p0), dev(r0)
    with T.Tvfgp(nx, ny, nz) as h:
        t_ref = h.run(bd, p_ref, r_ref, lam, 7, 1.0)
        t_ref = h.run(bd, p_ref, r_ref, lam, 4, t_ref)
        assert h.check() == T.TVFGP_OK

    # a first call on other buffers, so that module loading and the
    # address lookup are behind us when free memory is measured
    pw, rw = dev(p0), dev(r0)
    tf = ctypes.c_double(0.0)
    assert fn(nx, ny, nz, bd.data_ptr(), pw.data_ptr(), rw.data_ptr(), lam, 1, 1.0, stream,
              ctypes.byref(tf)) == T.TVFGP_OK
    torch.cuda.synchronize()

    # the entry point that allocates nothing: two calls in a row
    p, r = dev(p0), dev(r0)
    free_before = torch.cuda.mem_get_info()[0]
    assert fn(nx, ny, nz, bd.data_ptr(), p.data_ptr(), r.data_ptr(), lam, 7, 1.0, stream,
              ctypes.byref(tf)) == T.TVFGP_OK
    t1 = tf.value
    assert fn(nx, ny, nz, bd.data_ptr(), p.data_ptr(), r.data_ptr(), lam, 4, t1, stream,
              ctypes.byref(tf)) == T.TVFGP_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before

    assert t1 == t1o and tf.value == t2o == t_ref
    ph, rh = p.cpu().numpy(), r.cpu().numpy()
    dp = float(np.abs(ph - po).max())
    dr = float(np.abs(rh - ro).max())
    assert dp <= TOL and dr <= TOL, (dp, dr)
    assert np.array_equal(ph, po) and np.array_equal(rh, ro), "not bitwise equal to the oracle"
    assert torch.equal(p, p_ref) and torch.equal(r, r_ref), "not bitwise equal to tvfgp_run"


def test_noalloc_refuses_volumes_above_its_capacity():
    T, fn = c_entry()
    tf = ctypes.c_double(0.0)
    assert 129 * 128 * 128 > MAX_VOXELS
    rc = fn(129, 128, 128, None, None, None, 0.04, 3, 1.0, None, ctypes.byref(tf))
    assert rc == T.TVFGP_ERR_UNSUPPORTED
    rc = fn(0, 4, 4, None, None, None, 0.04, 3, 1.0, None, ctypes.byref(tf))
    assert rc == T.TVFGP_ERR_ARG


def test_noalloc_refuses_buffers_inside_its_array():
    import torch
    T, fn = c_entry()
    addr, size = T.tvfgp_debug_noalloc_scratch()
    assert addr != 0 and size == 3 * 4 * MAX_VOXELS
    shape = (16, 8, 4)
    n = 16 * 8 * 4
    b = dev(synth.random_case(shape, 31))
    p = dev(synth.random_dual(shape, 32, scale=0.3))
    r = dev(synth.random_dual(shape, 33, scale=0.3))
    before = (p.clone(), r.clone())
    tf = ctypes.c_double(0.0)
    stream = torch.cuda.current_stream().cuda_stream
    inside = [addr, addr + size - 4 * 3 * n, addr + 4096]
    for a in inside:
        for args in ((a, p.data_ptr(), r.data_ptr()), (b.data_ptr(), a, r.data_ptr()),
                     (b.data_ptr(), p.data_ptr(), a)):
            assert fn(16, 8, 4, *args, 0.05, 3, 1.0, stream, ctypes.byref(tf)) == T.TVFGP_ERR_ARG
    torch.cuda.synchronize()
    assert torch.equal(p, before[0]) and torch.equal(r, before[1])


@pytest.mark.parametrize("shape", [(36, 13, 9), (5, 3, 7)])
def test_noalloc_writes_nothing_outside_the_buffers(shape):
    """Guard bands with a NaN canary around b, p and r; two calls in a row
    (vector kernel for nx % 4 == 0, scalar kernel otherwise)."""
    from gpu_util import Guarded
    T, fn = c_entry()
    nx, ny, nz = shape
    b = synth.random_case(shape, 91)
    p0 = synth.random_dual(shape, 92, scale=0.4)
    r0 = synth.random_dual(shape, 93, scale=0.6)
    gb, gp, gr = Guarded(b), Guarded(p0), Guarded(r0)
    tf = ctypes.c_double(0.0)
    assert fn(nx, ny, nz, gb.t.data_ptr(), gp.t.data_ptr(), gr.t.data_ptr(), 0.07, 5, 1.0, None,
              ctypes.byref(tf)) == T.TVFGP_OK
    assert fn(nx, ny, nz, gb.t.data_ptr(), gp.t.data_ptr(), gr.t.data_ptr(), 0.07, 2, tf.value, None,
              ctypes.byref(tf)) == T.TVFGP_OK
    for name, g in (("b", gb), ("p", gp), ("r", gr)):
        assert g.intact(), "%s: a canary was overwritten (%s)" % (name, shape)
    po, ro = p0.copy(), r0.copy()
    t = oracle.fgp_run(b, po, ro, 0.07, 5, 1.0)
    oracle.fgp_run(b, po, ro, 0.07, 2, t)
    assert np.array_equal(gp.values().view(np.float32), po.reshape(-1))
    assert np.array_equal(gr.values().view(np.float32), ro.reshape(-1))


CAPTURE_FIRST = r"""
import ctypes, sys
import torch
sys.path.insert(0, %r)
from fgp_dual_stencil_gb300 import tvfgp as T
lib = ctypes.CDLL(T.LIB_PATH)
fn = lib.tvfgp_run_noalloc
vp, i = ctypes.c_void_p, ctypes.c_int
fn.argtypes = [i, i, i, vp, vp, vp, ctypes.c_float, i, ctypes.c_double, vp, ctypes.POINTER(ctypes.c_double)]
fn.restype = i
b = torch.rand((4, 8, 16), device="cuda")
p = torch.zeros((3, 4, 8, 16), device="cuda")
r = torch.zeros_like(p)
torch.cuda.synchronize()
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
tf = ctypes.c_double(0.0)
with torch.cuda.graph(g, stream=s):
    rc = fn(16, 8, 4, b.data_ptr(), p.data_ptr(), r.data_ptr(), 0.05, 3, 1.0, s.cuda_stream, ctypes.byref(tf))
print("rc", rc)
"""


def test_noalloc_first_call_under_capture_is_refused():
    """In a fresh process, the first call comes while its stream is being
    captured: it must return TVFGP_ERR_ARG without looking up the array."""
    from fgp_dual_stencil_gb300 import tvfgp as T
    out = subprocess.run([sys.executable, "-c", CAPTURE_FIRST % ROOT], cwd=ROOT, capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert "rc %d" % T.TVFGP_ERR_ARG in out.stdout, out.stdout
