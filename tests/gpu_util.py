"""Helpers shared by the GPU tests: run a workload through the CUDA library
and through the CPU oracle on the same seeded inputs."""
import numpy as np

import oracle
from fgp_dual_stencil_gb300 import synth

# Parity bar: max abs diff <= 1e-5 on p and r, <= 1e-5 * max|b| on z.
TOL_DUAL = 1e-5
TOL_Z_REL = 1e-5


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def run_workload_gpu(w, variant="auto", graph=False, p0=None, r0=None):
    """The workload's outer loop (fresh b per outer, t0 per outer, p and r
    carried over) on the GPU.  Returns numpy (b_last, p, r, z_of_p, z_of_r)."""
    import torch
    from fgp_dual_stencil_gb300 import tvfgp as T
    base = synth.phantom(w)
    shape = (3, w.nz, w.ny, w.nx)
    p = dev(p0) if p0 is not None else torch.zeros(shape, device="cuda")
    r = dev(r0) if r0 is not None else torch.zeros(shape, device="cuda")
    with T.Tvfgp(w.nx, w.ny, w.nz, variant, graph) as h:
        b = None
        for k in range(w.outers):
            b_np = synth.make_b(w, k, base)
            b = dev(b_np)
            h.run(b, p, r, w.lam, w.steps, w.t0)
        zp = h.primal(b, p, w.lam)
        zr = h.primal(b, r, w.lam)
        assert h.check() == T.TVFGP_OK
        launched = h.launch_count
    torch.cuda.synchronize()
    return b_np, host(p), host(r), host(zp), host(zr), launched


_ORACLE_RUNS = {}


def run_workload_oracle(w, p0=None, r0=None):
    """The workload on the oracle: (b_last, p, r, z_of_p, z_of_r).  Runs from
    p = r = 0 are computed once per test session and shared (the arrays are
    only read by the callers)."""
    if p0 is None and r0 is None:
        if w.key not in _ORACLE_RUNS:
            _ORACLE_RUNS[w.key] = _run_workload_oracle(w)
        return _ORACLE_RUNS[w.key]
    return _run_workload_oracle(w, p0, r0)


def _run_workload_oracle(w, p0=None, r0=None):
    base = synth.phantom(w)
    shape = (3, w.nz, w.ny, w.nx)
    p = np.zeros(shape, np.float32) if p0 is None else p0.copy()
    r = np.zeros(shape, np.float32) if r0 is None else r0.copy()
    b = None
    for k in range(w.outers):
        b = synth.make_b(w, k, base)
        oracle.fgp_run(b, p, r, w.lam, w.steps, w.t0)
    return b, p, r, oracle.primal(b, p, w.lam), oracle.primal(b, r, w.lam)


def max_diff(a, b):
    return float(np.abs(a.astype(np.float64) - b.astype(np.float64)).max()) if a.size else 0.0


def assert_parity(gpu, ref, bmax, exact=False, what=""):
    """gpu, ref: (p, r, z_p, z_r).  Checks the tolerance bar, and equality of
    values when exact is set."""
    names = ("p", "r", "z(p)", "z(r)")
    tols = (TOL_DUAL, TOL_DUAL, TOL_Z_REL * bmax, TOL_Z_REL * bmax)
    for name, g, o, tol in zip(names, gpu, ref, tols):
        d = max_diff(g, o)
        assert d <= tol, "%s %s: max abs diff %.3g > %.3g" % (what, name, d, tol)
        if exact:
            assert d == 0.0, "%s %s: not equal to the oracle (max abs diff %.3g)" % (what, name, d)


GUARD = 16384                                    # elements on each side
CANARY = np.uint32(0x7FC0BEEF)


class Guarded:
    """A CUDA buffer of n elements inside canary margins (GUARD elements of
    CANARY, a quiet NaN with a payload, on each side)."""

    def __init__(self, values, dtype_bits=32):
        import torch
        flat = np.ascontiguousarray(values).reshape(-1)
        self.n = flat.size
        word = np.uint16 if dtype_bits == 16 else np.uint32
        canary = word(0x7E5F) if dtype_bits == 16 else CANARY
        host = np.full(self.n + 2 * GUARD, canary, dtype=word)
        host[GUARD:GUARD + self.n] = flat.view(word)
        self.all = torch.from_numpy(host.view(np.int16 if dtype_bits == 16 else np.int32)).cuda()
        self.view_dtype = torch.float16 if dtype_bits == 16 else torch.float32
        self.canary = canary
        self.word = word

    @property
    def t(self):
        return self.all[GUARD:GUARD + self.n].view(self.view_dtype)

    def intact(self):
        host = self.all.cpu().numpy().view(self.word)
        return bool((host[:GUARD] == self.canary).all() and (host[GUARD + self.n:] == self.canary).all())

    def values(self):
        return self.all.cpu().numpy().view(self.word)[GUARD:GUARD + self.n]
