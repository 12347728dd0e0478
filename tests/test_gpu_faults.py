"""Failures injected on the host (no GPU fault): device allocations that
fail (tvfgp_debug_fail_allocs) at every allocation site, and handles that
are not handles.  Each must give a clean error code, leave no half-built
handle or leaked memory behind, and leave the state that was there
usable."""
import ctypes

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
    yield tvfgp
    tvfgp.tvfgp_debug_fail_allocs(0, 0)


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def create(T, shape, variant):
    h = ctypes.c_void_p(12345)
    rc = T.raw_call("tvfgp_create_ex", *shape, variant, 0, ctypes.byref(h))
    return rc, h.value


def small_run_matches_oracle(T, h, shape, nsteps=5):
    b = synth.random_case(shape, 7)
    p = dev(np.zeros((3,) + b.shape, np.float32))
    r = dev(np.zeros((3,) + b.shape, np.float32))
    T.tvfgp_run(h, dev(b), p, r, 0.05, nsteps)
    assert T.tvfgp_check(h) == T.TVFGP_OK
    po = np.zeros((3,) + b.shape, np.float32)
    ro = np.zeros_like(po)
    oracle.fgp_run(b, po, ro, 0.05, nsteps, 1.0)
    return np.array_equal(p.cpu().numpy(), po) and np.array_equal(r.cpu().numpy(), ro)


@pytest.mark.parametrize("skip", [0, 1, 2])
def test_create_fails_cleanly_at_each_allocation(T, skip):
    """AUTO handles allocate the scratch dual, the error word and the two
    extra dual sets of the two-step runs, in that order."""
    shape = (64, 32, 16)
    T.tvfgp_debug_fail_allocs(skip, 1)
    rc, h = create(T, shape, T.TVFGP_VARIANT_AUTO)
    T.tvfgp_debug_fail_allocs(0, 0)
    assert rc == T.TVFGP_ERR_OOM and h is None
    rc, h = create(T, shape, T.TVFGP_VARIANT_AUTO)
    assert rc == T.TVFGP_OK
    try:
        assert small_run_matches_oracle(T, h, shape)
    finally:
        T.tvfgp_destroy(h)


def test_failed_creates_leak_nothing(T):
    import torch
    shape = (256, 128, 64)                      # 24 MiB of scratch dual, 72 MiB of extra sets
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for k in range(6):
        T.tvfgp_debug_fail_allocs(1 + k % 2, 1)
        rc, h = create(T, shape, T.TVFGP_VARIANT_AUTO)
        assert rc == T.TVFGP_ERR_OOM and h is None
    T.tvfgp_debug_fail_allocs(0, 0)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free0 - free1 < 16 * 2**20, "failed creates kept %d bytes" % (free0 - free1)


@pytest.mark.parametrize("target", ["zmarch2", "separate"])
def test_set_variant_oom_keeps_the_handle(T, target):
    shape = (32, 16, 16)
    rc, h = create(T, shape, T.TVFGP_VARIANT_FUSED)
    assert rc == T.TVFGP_OK
    try:
        T.tvfgp_debug_fail_allocs(0, 1)
        rc = T.raw_call("tvfgp_set_variant", h, T.VARIANTS[target])
        T.tvfgp_debug_fail_allocs(0, 0)
        assert rc == T.TVFGP_ERR_OOM
        assert small_run_matches_oracle(T, h, shape)
        assert T.tvfgp_last_variant(h) == T.TVFGP_VARIANT_FUSED      # the variant did not change
        T.tvfgp_set_variant(h, target)                              # and can be set afterwards
        assert small_run_matches_oracle(T, h, shape)
    finally:
        T.tvfgp_destroy(h)


@pytest.mark.parametrize("skip", [0, 1])
def test_packed_run_oom_runs_in_place(T, skip):
    """A long run on padded rows whose dense staging (skip 0) or dense
    shadow handle (skip 1) cannot be allocated runs in place instead."""
    import torch
    shape = (32, 12, 10)
    nx, ny, nz = shape
    pitch = T.fft_pitch(nx)
    b = synth.random_case(shape, 8)
    bp = np.zeros(b.shape[:-1] + (pitch,), np.float32)
    bp[..., :nx] = b
    p = torch.zeros((3, nz, ny, pitch), device="cuda")
    r = torch.zeros_like(p)
    with T.Tvfgp(nx, ny, nz, pitch=pitch) as h:
        T.tvfgp_debug_fail_allocs(skip, 1)
        h.run(dev(bp), p, r, 0.05, 6)
        T.tvfgp_debug_fail_allocs(0, 0)
        assert h.last_variant == T.TVFGP_VARIANT_FUSED
        assert h.check() == 0
        po = np.zeros((3,) + b.shape, np.float32)
        ro = np.zeros_like(po)
        oracle.fgp_run(b, po, ro, 0.05, 6, 1.0)
        assert np.array_equal(p.cpu().numpy()[..., :nx], po)
        assert np.array_equal(r.cpu().numpy()[..., :nx], ro)
        # the next long run packs
        h.run(dev(bp), p, r, 0.05, 6)
        assert h.last_variant == T.TVFGP_VARIANT_ZMARCH2_TMA


def test_not_a_handle(T):
    """A pointer to memory that is not a handle is rejected by every call."""
    fake = (ctypes.c_int * 64)()
    h = ctypes.addressof(fake)
    tf = ctypes.c_double()
    assert T.raw_call("tvfgp_run", h, None, None, None, ctypes.c_float(0.1), 1, ctypes.c_double(1.0), None,
                      ctypes.byref(tf)) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_check", h, None) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_set_graph", h, 1) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_destroy", h) == T.TVFGP_ERR_ARG
    assert T.tvfgp_last_variant(h) == -1
