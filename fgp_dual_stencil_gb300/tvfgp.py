"""Python binding of libtvfgp.so (C ABI in include/tvfgp.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library.  Functions keep the C names.  Buffers are torch CUDA
float32 contiguous tensors (or raw device addresses as ints): a scalar volume
has nx*ny*nz elements (shape (nz, ny, nx) by convention), a dual field 3x that
(shape (3, nz, ny, nx)).  ``stream`` is a torch.cuda.Stream, a raw
cudaStream_t as int, or None for torch's current stream.

If libtvfgp.so has not been built, importing this module raises ImportError:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtvfgp.so")

TVFGP_OK = 0
TVFGP_ERR_ARG = 1
TVFGP_ERR_ALIGN = 2
TVFGP_ERR_CUDA = 3
TVFGP_ERR_OOM = 4
TVFGP_ERR_TIMEOUT = 5
TVFGP_ERR_UNSUPPORTED = 6

TVFGP_VARIANT_AUTO = 0
TVFGP_VARIANT_FUSED = 1
TVFGP_VARIANT_SCALAR = 2
TVFGP_VARIANT_ZMARCH_TMA = 3
TVFGP_VARIANT_ZMARCH2_TMA = 4
TVFGP_VARIANT_SEPARATE = 5
TVFGP_VARIANT_CUBE_TMA = 6

VARIANTS = {"auto": TVFGP_VARIANT_AUTO, "fused": TVFGP_VARIANT_FUSED,
            "scalar": TVFGP_VARIANT_SCALAR, "zmarch": TVFGP_VARIANT_ZMARCH_TMA,
            "zmarch2": TVFGP_VARIANT_ZMARCH2_TMA, "separate": TVFGP_VARIANT_SEPARATE,
            "cube": TVFGP_VARIANT_CUBE_TMA}


class TvfgpError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s failed: %s (status %d)" % (where, strerror(code), code))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libtvfgp.so is not built (%s); run `python -m "
                          "fgp_dual_stencil_gb300._build` or __graft_entry__.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    i, u, d, f, vp, ll = (ctypes.c_int, ctypes.c_uint, ctypes.c_double, ctypes.c_float,
                          ctypes.c_void_p, ctypes.c_longlong)
    sig = {
        "tvfgp_create": ([i, i, i, ctypes.POINTER(vp)], i),
        "tvfgp_create_ex": ([i, i, i, i, u, ctypes.POINTER(vp)], i),
        "tvfgp_create_pitched": ([i, i, i, i, ctypes.POINTER(vp)], i),
        "tvfgp_destroy": ([vp], i),
        "tvfgp_set_variant": ([vp, i], i),
        "tvfgp_set_graph": ([vp, i], i),
        "tvfgp_run": ([vp, vp, vp, vp, f, i, d, vp, ctypes.POINTER(d)], i),
        "tvfgp_step": ([vp, vp, vp, vp, vp, f, f, vp], i),
        "tvfgp_primal": ([vp, vp, vp, f, vp, vp], i),
        "tvfgp_momentum": ([d, i, ctypes.POINTER(d), ctypes.POINTER(d)], i),
        "tvfgp_check": ([vp, vp], i),
        "tvfgp_last_variant": ([vp], i),
        "tvfgp_launch_count": ([vp], ll),
        "tvfgp_debug_timeout_probe": ([vp, i, vp], i),
        "tvfgp_debug_set_poll_limit": ([vp, i, i], i),
        "tvfgp_debug_fail_allocs": ([i, i], i),
        "tvfgp_debug_plan": ([i, i, i, i, i, i, d, ctypes.POINTER(i), ctypes.POINTER(i), ctypes.POINTER(i),
                              ctypes.POINTER(f), i, ctypes.POINTER(i)], i),
        "tvfgp_debug_chunks": ([i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i), ctypes.POINTER(i), i,
                                ctypes.POINTER(i)], i),
        "tvfgp_debug_projection_check": ([i, ctypes.c_ulonglong, ctypes.c_ulonglong, vp, vp], i),
        "tvfgp_run_noalloc": ([i, i, i, vp, vp, vp, f, i, d, vp, ctypes.POINTER(d)], i),
        "tvfgp_debug_noalloc_scratch": ([ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_ulonglong)], i),
        "tvfgp_host_alloc": ([ctypes.c_size_t, i, ctypes.POINTER(vp)], i),
        "tvfgp_run_f16": ([vp, vp, vp, vp, f, i, d, vp, ctypes.POINTER(d)], i),
        "tvfgp_primal_f16": ([vp, vp, vp, f, vp, vp], i),
        "tvfgp_host_free": ([vp], i),
        "tvfgp_strerror": ([i], ctypes.c_char_p),
        "tvfgp_version": ([], i),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def _ok(code: int, where: str) -> None:
    if code != TVFGP_OK:
        raise TvfgpError(code, where)


def _addr(x, n: int | None, name: str):
    """Device address of a torch tensor (checked) or a raw int address."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch
    if not isinstance(x, torch.Tensor):
        raise TypeError("%s must be a torch tensor or an int address" % name)
    if not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("%s must be a contiguous float32 CUDA tensor" % name)
    if n is not None and x.numel() != n:
        raise ValueError("%s has %d elements, expected %d" % (name, x.numel(), n))
    return x.data_ptr()


def _addr16(x, n: int | None, name: str):
    """Device address of a torch float16 CUDA tensor (the binary16 dual)."""
    if x is None or isinstance(x, int):
        return x
    import torch
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float16 \
            or not x.is_contiguous():
        raise ValueError("%s must be a contiguous float16 CUDA tensor" % name)
    if n is not None and x.numel() != n:
        raise ValueError("%s has %d elements, expected %d" % (name, x.numel(), n))
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def strerror(code: int) -> str:
    return _lib.tvfgp_strerror(int(code)).decode()


def tvfgp_version() -> int:
    return int(_lib.tvfgp_version())


def tvfgp_strerror(code: int) -> str:
    return strerror(code)


def tvfgp_momentum(t0: float, nsteps: int):
    """(list of m_k, t after the last step), computed by the library's host code."""
    m = (ctypes.c_double * max(int(nsteps), 1))()
    tf = ctypes.c_double(0.0)
    _ok(_lib.tvfgp_momentum(float(t0), int(nsteps), m, ctypes.byref(tf)), "tvfgp_momentum")
    return [m[k] for k in range(int(nsteps))], tf.value


def tvfgp_create(nx: int, ny: int, nz: int, variant: int | str = TVFGP_VARIANT_AUTO,
                 flags: int = 0) -> int:
    """Create a handle (an opaque int) for an nx x ny x nz volume."""
    if isinstance(variant, str):
        variant = VARIANTS[variant]
    h = ctypes.c_void_p()
    _ok(_lib.tvfgp_create_ex(int(nx), int(ny), int(nz), int(variant), int(flags), ctypes.byref(h)),
        "tvfgp_create")
    return h.value


def tvfgp_create_pitched(nx: int, ny: int, nz: int, pitch: int) -> int:
    """Create a handle for volumes whose rows hold `pitch` elements (x < nx
    used), e.g. pitch = 2 * (nx // 2 + 1), the in-place real-to-complex FFT
    layout."""
    h = ctypes.c_void_p()
    _ok(_lib.tvfgp_create_pitched(int(nx), int(ny), int(nz), int(pitch), ctypes.byref(h)),
        "tvfgp_create_pitched")
    return h.value


def fft_pitch(nx: int) -> int:
    """Row pitch of an in-place real-to-complex FFT of length nx: 2*(nx/2+1)."""
    return 2 * (int(nx) // 2 + 1)


def tvfgp_destroy(h: int) -> None:
    _ok(_lib.tvfgp_destroy(h), "tvfgp_destroy")


def tvfgp_set_variant(h: int, variant: int | str) -> None:
    if isinstance(variant, str):
        variant = VARIANTS[variant]
    _ok(_lib.tvfgp_set_variant(h, int(variant)), "tvfgp_set_variant")


def tvfgp_set_graph(h: int, enable: bool) -> None:
    _ok(_lib.tvfgp_set_graph(h, 1 if enable else 0), "tvfgp_set_graph")


def tvfgp_run(h: int, b, p, r, lam: float, nsteps: int, t0: float = 1.0, stream=None,
              n: int | None = None) -> float:
    """nsteps FGP steps on (p, r) in place; returns t after the last step."""
    tf = ctypes.c_double(0.0)
    _ok(_lib.tvfgp_run(h, _addr(b, n, "b"), _addr(p, None if n is None else 3 * n, "p"),
                       _addr(r, None if n is None else 3 * n, "r"), float(lam), int(nsteps),
                       float(t0), _stream(stream), ctypes.byref(tf)), "tvfgp_run")
    return tf.value


def tvfgp_step(h: int, b, p, r_src, r_dst, lam: float, m: float, stream=None) -> None:
    """One step with explicit momentum weight and ping-pong buffers."""
    _ok(_lib.tvfgp_step(h, _addr(b, None, "b"), _addr(p, None, "p"), _addr(r_src, None, "r_src"),
                        _addr(r_dst, None, "r_dst"), float(lam), float(m), _stream(stream)),
        "tvfgp_step")


def tvfgp_primal(h: int, b, dual, lam: float, z, stream=None) -> None:
    """z = max(b - lam * L(dual), 0)."""
    _ok(_lib.tvfgp_primal(h, _addr(b, None, "b"), _addr(dual, None, "dual"), float(lam),
                          _addr(z, None, "z"), _stream(stream)), "tvfgp_primal")


def tvfgp_run_f16(h: int, b, p16, r16, lam: float, nsteps: int, t0: float = 1.0, stream=None,
                  n: int | None = None) -> float:
    """tvfgp_run with p and r stored as float16 tensors; returns t after the last step."""
    tf = ctypes.c_double(0.0)
    _ok(_lib.tvfgp_run_f16(h, _addr(b, n, "b"), _addr16(p16, None if n is None else 3 * n, "p"),
                           _addr16(r16, None if n is None else 3 * n, "r"), float(lam), int(nsteps),
                           float(t0), _stream(stream), ctypes.byref(tf)), "tvfgp_run_f16")
    return tf.value


def tvfgp_primal_f16(h: int, b, dual16, lam: float, z, stream=None) -> None:
    _ok(_lib.tvfgp_primal_f16(h, _addr(b, None, "b"), _addr16(dual16, None, "dual"), float(lam),
                              _addr(z, None, "z"), _stream(stream)), "tvfgp_primal_f16")


def tvfgp_check(h: int, stream=None) -> int:
    """Synchronise the stream and return the status of the device error word
    (TVFGP_OK or TVFGP_ERR_TIMEOUT); raises on CUDA errors."""
    code = int(_lib.tvfgp_check(h, _stream(stream)))
    if code not in (TVFGP_OK, TVFGP_ERR_TIMEOUT):
        raise TvfgpError(code, "tvfgp_check")
    return code


def tvfgp_last_variant(h: int) -> int:
    return int(_lib.tvfgp_last_variant(h))


def tvfgp_launch_count(h: int) -> int:
    return int(_lib.tvfgp_launch_count(h))


def tvfgp_debug_projection_check(mode: int, count: int, seed: int, out, stream=None) -> None:
    """Enqueue the projection self-check (see the header); out is an int64
    CUDA tensor of 2 elements set to (0, -1) by the caller."""
    import torch
    if not isinstance(out, torch.Tensor) or not out.is_cuda or out.dtype != torch.int64 or out.numel() != 2:
        raise ValueError("out must be a CUDA int64 tensor of 2 elements")
    _ok(_lib.tvfgp_debug_projection_check(int(mode), int(count), int(seed) & (2**64 - 1), out.data_ptr(),
                                          _stream(stream)), "tvfgp_debug_projection_check")


def tvfgp_debug_fail_allocs(skip: int, count: int) -> None:
    """Let the library's next `skip` device allocations succeed and fail the
    `count` after them (test hook; count = 0 clears it)."""
    _ok(_lib.tvfgp_debug_fail_allocs(int(skip), int(count)), "tvfgp_debug_fail_allocs")


def tvfgp_debug_plan(nx: int, ny: int, nz: int, pitch: int = 0, variant: int | str = TVFGP_VARIANT_AUTO,
                     nsteps: int = 1, t0: float = 1.0):
    """The launches tvfgp_run would enqueue (host only, no GPU): returns
    (route, copy_back, launches), each launch a dict with the variant, the
    buffer roles of b, p_src, p_dst, r_src, r_dst, its flags and its two
    momentum weights (see tvfgp.h)."""
    v = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    route, copy_back, count = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _ok(_lib.tvfgp_debug_plan(nx, ny, nz, pitch, v, nsteps, float(t0), ctypes.byref(route),
                              ctypes.byref(copy_back), None, None, 0, ctypes.byref(count)), "tvfgp_debug_plan")
    n = count.value
    items = (ctypes.c_int * max(7 * n, 1))()
    m = (ctypes.c_float * max(2 * n, 1))()
    _ok(_lib.tvfgp_debug_plan(nx, ny, nz, pitch, v, nsteps, float(t0), ctypes.byref(route),
                              ctypes.byref(copy_back), items, m, n, ctypes.byref(count)), "tvfgp_debug_plan")
    keys = ("variant", "b", "p_src", "p_dst", "r_src", "r_dst", "flags")
    launches = [dict(zip(keys, items[7 * k:7 * k + 7]), m=(m[2 * k], m[2 * k + 1])) for k in range(n)]
    return route.value, bool(copy_back.value), launches


def tvfgp_debug_chunks(nx: int, ny: int, nz: int, slots: int):
    """(zc, [(z0, ze), ...]): the two-step kernel's split of the planes among
    its CTAs with `slots` resident CTAs (host only, no GPU)."""
    zc, count = ctypes.c_int(), ctypes.c_int()
    _ok(_lib.tvfgp_debug_chunks(nx, ny, nz, slots, ctypes.byref(zc), None, None, 0, ctypes.byref(count)),
        "tvfgp_debug_chunks")
    n = count.value
    z0, ze = (ctypes.c_int * max(n, 1))(), (ctypes.c_int * max(n, 1))()
    _ok(_lib.tvfgp_debug_chunks(nx, ny, nz, slots, ctypes.byref(zc), z0, ze, n, ctypes.byref(count)),
        "tvfgp_debug_chunks")
    return zc.value, [(z0[j], ze[j]) for j in range(n)]


def tvfgp_debug_timeout_probe(h: int, spins: int, stream=None) -> None:
    _ok(_lib.tvfgp_debug_timeout_probe(h, int(spins), _stream(stream)), "tvfgp_debug_timeout_probe")


def tvfgp_debug_set_poll_limit(h: int, polls: int, from_plane: int = 0) -> None:
    """Polls each wait for data of the TMA kernels makes before giving up
    (0: at once; < 0: the default), for each CTA's planes from from_plane on.
    Test hook; no work of h in flight."""
    _ok(_lib.tvfgp_debug_set_poll_limit(h, int(polls), int(from_plane)), "tvfgp_debug_set_poll_limit")


TVFGP_NOALLOC_MAX_VOXELS = 2097152


def tvfgp_run_noalloc(nx: int, ny: int, nz: int, b, p, r, lam: float, nsteps: int,
                      t0: float = 1.0, stream=None) -> float:
    """tvfgp_run with no handle and no allocation (for callers that may not
    allocate device memory); at most TVFGP_NOALLOC_MAX_VOXELS voxels, and
    calls that overlap on the GPU must be serialised by the caller.  Returns
    t after the last step."""
    n = int(nx) * int(ny) * int(nz)
    tf = ctypes.c_double(0.0)
    _ok(_lib.tvfgp_run_noalloc(int(nx), int(ny), int(nz), _addr(b, n, "b"), _addr(p, 3 * n, "p"),
                               _addr(r, 3 * n, "r"), float(lam), int(nsteps), float(t0),
                               _stream(stream), ctypes.byref(tf)), "tvfgp_run_noalloc")
    return tf.value


def tvfgp_host_alloc(nbytes: int, write_combined: bool = False) -> int:
    """Page-locked host memory (an int address); see include/tvfgp.h."""
    p = ctypes.c_void_p()
    _ok(_lib.tvfgp_host_alloc(int(nbytes), 1 if write_combined else 0, ctypes.byref(p)),
        "tvfgp_host_alloc")
    return p.value


def tvfgp_host_free(addr: int) -> None:
    _ok(_lib.tvfgp_host_free(addr), "tvfgp_host_free")


def host_tensor(shape, write_combined: bool = False):
    """A float32 CPU torch tensor of `shape` over tvfgp_host_alloc memory,
    freed when the tensor (and any view of it) is garbage collected.
    Write-combined memory suits host-to-device inputs: fast to fill, slow to
    read back on the CPU."""
    import weakref
    import numpy as np
    import torch
    n = 1
    for s_ in shape:
        n *= int(s_)
    addr = tvfgp_host_alloc(4 * n, write_combined)
    arr = np.ctypeslib.as_array((ctypes.c_float * n).from_address(addr)).reshape(tuple(shape))
    weakref.finalize(arr, _lib.tvfgp_host_free, addr)
    return torch.from_numpy(arr)


def tvfgp_debug_noalloc_scratch() -> tuple[int, int]:
    """(device address, bytes) of tvfgp_run_noalloc's built-in array on the
    current device (test hook)."""
    addr, size = ctypes.c_void_p(), ctypes.c_ulonglong()
    _ok(_lib.tvfgp_debug_noalloc_scratch(ctypes.byref(addr), ctypes.byref(size)),
        "tvfgp_debug_noalloc_scratch")
    return int(addr.value or 0), int(size.value)


def raw_call(name: str, *args) -> int:
    """Call a C entry point with raw arguments and return its status code
    (for tests of the argument checks)."""
    return int(getattr(_lib, name)(*args))


class Tvfgp:
    """Owns one handle.  Tensors: b (nz, ny, nx), p and r (3, nz, ny, nx); with
    a row pitch, b (nz, ny, pitch) and p, r (3, nz, ny, pitch), of which only
    x < nx is read or written."""

    def __init__(self, nx: int, ny: int, nz: int, variant: int | str = TVFGP_VARIANT_AUTO,
                 graph: bool = False, pitch: int | None = None):
        self.shape = (int(nx), int(ny), int(nz))
        self.pitch = int(nx) if pitch is None else int(pitch)
        self.n = self.pitch * int(ny) * int(nz)
        if pitch is None:
            self.h = tvfgp_create(nx, ny, nz, variant)
        else:
            self.h = tvfgp_create_pitched(nx, ny, nz, pitch)
            if variant not in (TVFGP_VARIANT_AUTO, "auto"):
                tvfgp_set_variant(self.h, variant)
        if graph:
            tvfgp_set_graph(self.h, True)

    def run(self, b, p, r, lam, nsteps, t0=1.0, stream=None) -> float:
        return tvfgp_run(self.h, b, p, r, lam, nsteps, t0, stream, n=self.n)

    def step(self, b, p, r_src, r_dst, lam, m, stream=None) -> None:
        tvfgp_step(self.h, b, p, r_src, r_dst, lam, m, stream)

    def primal(self, b, dual, lam, z=None, stream=None):
        if z is None:
            import torch
            z = torch.empty_like(b)
        tvfgp_primal(self.h, b, dual, lam, z, stream)
        return z

    def run_f16(self, b, p16, r16, lam, nsteps, t0=1.0, stream=None) -> float:
        return tvfgp_run_f16(self.h, b, p16, r16, lam, nsteps, t0, stream, n=self.n)

    def primal_f16(self, b, dual16, lam, z=None, stream=None):
        if z is None:
            import torch
            z = torch.empty_like(b)
        tvfgp_primal_f16(self.h, b, dual16, lam, z, stream)
        return z

    def set_variant(self, v) -> None:
        tvfgp_set_variant(self.h, v)

    def set_graph(self, on: bool) -> None:
        tvfgp_set_graph(self.h, on)

    def check(self, stream=None) -> int:
        return tvfgp_check(self.h, stream)

    @property
    def last_variant(self) -> int:
        return tvfgp_last_variant(self.h)

    @property
    def launch_count(self) -> int:
        return tvfgp_launch_count(self.h)

    def close(self) -> None:
        if self.h:
            tvfgp_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
