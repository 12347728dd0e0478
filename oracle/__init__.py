"""CPU oracle for the FGP step on the 3D isotropic TV dual.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow reference the GPU
path is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import it.  The library in
``fgp_dual_stencil_gb300`` never imports it, and it imports nothing from
there.

The arithmetic lives in ``tvfgp_oracle.c`` (plain C, no FMA contraction,
optional OpenMP over z-planes), which follows the page "TV solver: the FGP
step on the GPU", section "What one step does".  This module compiles it with
gcc on first use and marshals numpy arrays to it; it adds no arithmetic of its
own.

Array conventions (numpy, C order): a scalar volume has shape (nz, ny, nx), so
x is fastest; a dual field has shape (3, nz, ny, nx), component a = 0, 1, 2 for
the x, y, z axes.  dtype float32 selects the fp32 parity oracle, float64 its
fp64 twin.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "tvfgp_oracle.c"), os.path.join(_HERE, "tvfgp_oracle_body.h")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libtvfgp_oracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: gcc contracts a*b+c into an FMA by default on aarch64,
# which would change the rounding of the canonical expression order.
CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
          "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard"]


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/ (if missing or older than its
    sources) and return the path of the shared library."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest = max(os.path.getmtime(s) for s in _SRC)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC[0], "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c_int, c_dbl, vp = ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.oracle_momentum.argtypes = [c_dbl, c_int, vp, vp]
        lib.oracle_momentum.restype = None
        lib.oracle_set_threads.argtypes = [c_int]
        lib.oracle_get_threads.restype = c_int
        for suf, real in (("_f32", ctypes.c_float), ("_f64", ctypes.c_double)):
            f = getattr(lib, "oracle_adjoint" + suf)
            f.argtypes = [c_int, c_int, c_int, vp, vp]
            f.restype = None
            f = getattr(lib, "oracle_gradient" + suf)
            f.argtypes = [c_int, c_int, c_int, vp, vp]
            f.restype = None
            f = getattr(lib, "oracle_primal" + suf)
            f.argtypes = [c_int, c_int, c_int, vp, vp, real, vp]
            f.restype = None
            f = getattr(lib, "oracle_fgp_step" + suf)
            f.argtypes = [c_int, c_int, c_int, vp, vp, vp, vp, vp, real, real]
            f.restype = None
            f = getattr(lib, "oracle_fgp_run" + suf)
            f.argtypes = [c_int, c_int, c_int, vp, vp, vp, real, c_int, c_dbl, vp]
            f.restype = c_int
        lib.oracle_half_to_float.argtypes = [ctypes.c_ushort]
        lib.oracle_half_to_float.restype = ctypes.c_float
        lib.oracle_float_to_half.argtypes = [ctypes.c_float]
        lib.oracle_float_to_half.restype = ctypes.c_ushort
        for name in ("oracle_half_to_float_array", "oracle_float_to_half_array"):
            getattr(lib, name).argtypes = [vp, vp, ctypes.c_size_t]
            getattr(lib, name).restype = None
        lib.oracle_primal_h16.argtypes = [c_int, c_int, c_int, vp, vp, ctypes.c_float, vp]
        lib.oracle_primal_h16.restype = None
        lib.oracle_fgp_step_h16.argtypes = [c_int, c_int, c_int, vp, vp, vp, vp, ctypes.c_float,
                                            ctypes.c_float]
        lib.oracle_fgp_step_h16.restype = c_int
        lib.oracle_fgp_run_h16.argtypes = [c_int, c_int, c_int, vp, vp, vp, ctypes.c_float, c_int,
                                           c_dbl, vp]
        lib.oracle_fgp_run_h16.restype = c_int
        _lib = lib
        return lib


def _suffix(dtype) -> str:
    dt = np.dtype(dtype)
    if dt == np.float32:
        return "_f32"
    if dt == np.float64:
        return "_f64"
    raise TypeError("oracle arrays must be float32 or float64, got %s" % dt)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check_scalar(name, a, dtype=None):
    if not isinstance(a, np.ndarray) or a.ndim != 3:
        raise ValueError("%s must be a (nz, ny, nx) numpy array" % name)
    if not a.flags.c_contiguous:
        raise ValueError("%s must be C-contiguous" % name)
    if dtype is not None and a.dtype != dtype:
        raise TypeError("%s has dtype %s, expected %s" % (name, a.dtype, dtype))


def _check_dual(name, a, shape, dtype):
    if not isinstance(a, np.ndarray) or a.shape != (3,) + tuple(shape):
        raise ValueError("%s must have shape (3,)+%s" % (name, tuple(shape)))
    if not a.flags.c_contiguous or a.dtype != dtype:
        raise ValueError("%s must be C-contiguous %s" % (name, dtype))


def set_threads(n: int) -> None:
    """Set the OpenMP thread count of the oracle (results do not depend on it)."""
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def momentum(t0: float, nsteps: int):
    """Momentum weights m[0..nsteps-1] (float64) and t after the last step."""
    lib = _load()
    m = np.zeros(max(nsteps, 0), dtype=np.float64)
    tf = ctypes.c_double(0.0)
    lib.oracle_momentum(float(t0), int(max(nsteps, 0)), _ptr(m), ctypes.byref(tf))
    return m, tf.value if nsteps > 0 else float(t0)


def adjoint(dual: np.ndarray) -> np.ndarray:
    """L(dual)(j) = sum_a dual_a(j) - dual_a(j - e_a), zero below the lower faces."""
    shape = dual.shape[1:]
    _check_dual("dual", dual, shape, dual.dtype)
    out = np.empty(shape, dtype=dual.dtype)
    nz, ny, nx = shape
    getattr(_load(), "oracle_adjoint" + _suffix(dual.dtype))(nx, ny, nz, _ptr(dual), _ptr(out))
    return out


def gradient(z: np.ndarray) -> np.ndarray:
    """g_a(i) = z(i) - z(i + e_a), 0 where i + e_a leaves the volume; shape (3,)+z.shape."""
    _check_scalar("z", z)
    nz, ny, nx = z.shape
    g = np.empty((3,) + z.shape, dtype=z.dtype)
    getattr(_load(), "oracle_gradient" + _suffix(z.dtype))(nx, ny, nz, _ptr(z), _ptr(g))
    return g


def primal(b: np.ndarray, dual: np.ndarray, lam: float) -> np.ndarray:
    """z = max(b - lam * L(dual), 0)."""
    _check_scalar("b", b)
    _check_dual("dual", dual, b.shape, b.dtype)
    nz, ny, nx = b.shape
    z = np.empty_like(b)
    getattr(_load(), "oracle_primal" + _suffix(b.dtype))(nx, ny, nz, _ptr(b), _ptr(dual), lam, _ptr(z))
    return z


def fgp_step(b, p, r_src, lam, m):
    """One FGP step.  Updates p in place and returns (r_dst, z) where z is the
    primal of r_src that the step used."""
    _check_scalar("b", b)
    _check_dual("p", p, b.shape, b.dtype)
    _check_dual("r_src", r_src, b.shape, b.dtype)
    nz, ny, nx = b.shape
    r_dst = np.empty_like(r_src)
    zw = np.empty_like(b)
    getattr(_load(), "oracle_fgp_step" + _suffix(b.dtype))(
        nx, ny, nz, _ptr(b), _ptr(p), _ptr(r_src), _ptr(r_dst), _ptr(zw), lam, m)
    return r_dst, zw


def fgp_run(b, p, r, lam, nsteps, t0=1.0):
    """nsteps FGP steps; p and r are updated in place.  Returns t after the
    last step."""
    _check_scalar("b", b)
    _check_dual("p", p, b.shape, b.dtype)
    _check_dual("r", r, b.shape, b.dtype)
    nz, ny, nx = b.shape
    tf = ctypes.c_double(0.0)
    rc = getattr(_load(), "oracle_fgp_run" + _suffix(b.dtype))(
        nx, ny, nz, _ptr(b), _ptr(p), _ptr(r), lam, int(nsteps), float(t0), ctypes.byref(tf))
    if rc != 0:
        raise MemoryError("oracle could not allocate its work buffers")
    return tf.value


# ---------------------------------------------------------------------------
# binary16 storage of the dual (arrays of uint16 holding the IEEE bits)
# ---------------------------------------------------------------------------

def half_to_float(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().oracle_half_to_float_array(_ptr(h), _ptr(out), h.size)
    return out


def float_to_half(f: np.ndarray) -> np.ndarray:
    """Round float32 values to binary16 (nearest, ties to even); uint16 bits."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    _load().oracle_float_to_half_array(_ptr(f), _ptr(out), f.size)
    return out


def _check_dual16(name, a, shape):
    if not isinstance(a, np.ndarray) or a.shape != (3,) + tuple(shape) or a.dtype != np.uint16 \
            or not a.flags.c_contiguous:
        raise ValueError("%s must be a C-contiguous uint16 array of shape (3,)+%s" % (name, tuple(shape)))


def primal_h16(b, dual16, lam):
    _check_scalar("b", b, np.float32)
    _check_dual16("dual", dual16, b.shape)
    nz, ny, nx = b.shape
    z = np.empty_like(b)
    _load().oracle_primal_h16(nx, ny, nz, _ptr(b), _ptr(dual16), lam, _ptr(z))
    return z


def fgp_step_h16(b, p16, r_src16, lam, m):
    """One step with binary16 storage; p16 updated in place; returns r_dst16."""
    _check_scalar("b", b, np.float32)
    _check_dual16("p", p16, b.shape)
    _check_dual16("r_src", r_src16, b.shape)
    nz, ny, nx = b.shape
    r_dst = np.empty_like(r_src16)
    rc = _load().oracle_fgp_step_h16(nx, ny, nz, _ptr(b), _ptr(p16), _ptr(r_src16), _ptr(r_dst), lam, m)
    if rc != 0:
        raise MemoryError("oracle could not allocate its work buffers")
    return r_dst


def fgp_run_h16(b, p16, r16, lam, nsteps, t0=1.0):
    """nsteps steps with binary16 storage of p and r (updated in place)."""
    _check_scalar("b", b, np.float32)
    _check_dual16("p", p16, b.shape)
    _check_dual16("r", r16, b.shape)
    nz, ny, nx = b.shape
    tf = ctypes.c_double(0.0)
    rc = _load().oracle_fgp_run_h16(nx, ny, nz, _ptr(b), _ptr(p16), _ptr(r16), lam, int(nsteps),
                                    float(t0), ctypes.byref(tf))
    if rc != 0:
        raise MemoryError("oracle could not allocate its work buffers")
    return tf.value
