"""C-ABI library on a machine without a GPU: it builds, loads, exports every
declared entry point, and its host-only logic (argument checks, momentum
schedule, status strings) behaves as include/tvfgp.h states."""
import ctypes
import os
import re
import subprocess
import sys

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def T():
    from fgp_dual_stencil_gb300 import _build
    _build.build()
    from fgp_dual_stencil_gb300 import tvfgp
    return tvfgp


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(tvfgp_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(T):
    declared = declared_functions()
    assert {"tvfgp_create", "tvfgp_run", "tvfgp_primal", "tvfgp_destroy", "tvfgp_step"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", T.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (tvfgp_\w+)", out))
    assert declared <= exported, declared - exported
    lib = ctypes.CDLL(T.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name)


def test_no_oracle_code_in_the_library(T):
    out = subprocess.run(["nm", "-D", T.LIB_PATH], capture_output=True, text=True, check=True).stdout
    assert "oracle" not in out


def test_momentum_schedule_matches_oracle(T):
    for t0, n in ((1.0, 200), (2.75, 33), (1.0, 0)):
        m, tf = T.tvfgp_momentum(t0, n)
        mo, tfo = oracle.momentum(t0, n)
        assert np.array_equal(np.array(m, dtype=np.float64), mo) and tf == tfo
    with pytest.raises(T.TvfgpError):
        T.tvfgp_momentum(0.5, 3)
    with pytest.raises(T.TvfgpError):
        T.tvfgp_momentum(1.0, -1)


def test_create_rejects_bad_shapes_before_touching_cuda(T):
    h = ctypes.c_void_p()
    for dims in ((0, 4, 4), (4, -1, 4), (4, 4, 0), (70000, 1, 1), (65535, 65535, 1)):
        assert T.raw_call("tvfgp_create", *dims, ctypes.byref(h)) == T.TVFGP_ERR_ARG
        assert h.value is None
    assert T.raw_call("tvfgp_create_ex", 4, 4, 4, 7, 0, ctypes.byref(h)) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_create_ex", 4, 4, 4, 0, 1, ctypes.byref(h)) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_create", 4, 4, 4, None) == T.TVFGP_ERR_ARG
    # the size limit, a plane nx*ny <= 2^31 - 1, at its boundary; the volume
    # itself is bounded by device memory only (a GPU would allocate here)
    assert T.raw_call("tvfgp_create", 65535, 32769, 1, ctypes.byref(h)) == T.TVFGP_ERR_ARG
    for dims in ((65535, 32768, 1), (2048, 1024, 1025)):
        rc = T.raw_call("tvfgp_create", *dims, ctypes.byref(h))
        assert rc != T.TVFGP_ERR_ARG
        if rc == T.TVFGP_OK:
            T.raw_call("tvfgp_destroy", h)


def test_calls_on_a_null_handle(T):
    assert T.raw_call("tvfgp_destroy", None) == T.TVFGP_OK
    assert T.raw_call("tvfgp_set_graph", None, 1) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_set_variant", None, 1) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_check", None, None) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_last_variant", None) == -1
    assert T.raw_call("tvfgp_launch_count", None) == -1


def test_status_strings_and_version(T):
    assert T.tvfgp_version() >= 10000
    assert T.strerror(0) == "ok"
    seen = {T.strerror(c) for c in range(7)}
    assert len(seen) == 7
    assert T.strerror(99) == "unknown status code"


def test_create_without_a_gpu_reports_a_cuda_error(T):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert T.raw_call("tvfgp_create", 8, 8, 8, ctypes.byref(h)) in (T.TVFGP_ERR_CUDA, T.TVFGP_ERR_OOM)
    assert h.value is None


def test_host_alloc_argument_checks(T):
    p = ctypes.c_void_p(1)
    assert T.raw_call("tvfgp_host_alloc", 0, 0, ctypes.byref(p)) == T.TVFGP_ERR_ARG
    assert p.value is None
    assert T.raw_call("tvfgp_host_alloc", 16, 0, None) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_host_free", None) == T.TVFGP_OK


def test_allocation_failure_hook_without_gpu(T):
    """The allocation-failure hook fails a create cleanly before any device
    allocation is attempted; its arguments are checked."""
    assert T.raw_call("tvfgp_debug_fail_allocs", -1, 1) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_debug_fail_allocs", 0, -1) == T.TVFGP_ERR_ARG
    assert T.raw_call("tvfgp_debug_fail_allocs", 0, 1) == T.TVFGP_OK
    h = ctypes.c_void_p(5)
    try:
        assert T.raw_call("tvfgp_create", 8, 8, 8, ctypes.byref(h)) == T.TVFGP_ERR_OOM
        assert h.value is None
    finally:
        assert T.raw_call("tvfgp_debug_fail_allocs", 0, 0) == T.TVFGP_OK


def test_binding_fails_loudly_without_the_library():
    """With libtvfgp.so absent the binding raises ImportError at import; there
    is no fallback path."""
    code = (
        "import os, sys\n"
        "sys.path.insert(0, %r)\n"
        "real = os.path.exists\n"
        "os.path.exists = lambda p: False if str(p).endswith('libtvfgp.so') else real(p)\n"
        "try:\n"
        "    import fgp_dual_stencil_gb300.tvfgp\n"
        "except ImportError as e:\n"
        "    print('ImportError:', e)\n"
        "    sys.exit(0)\n"
        "sys.exit(3)\n" % ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "libtvfgp.so is not built" in out.stdout
