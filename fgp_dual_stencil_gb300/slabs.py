"""z-slab decomposition of the FGP step over several ranks (one GPU each).

The step (page "TV solver: the FGP step on the GPU", section "What one step
does") is local along z: at plane z it reads r of plane z-1 only through the
z difference of L, r_z(z) - r_z(z-1), and it reads the primal of plane z+1,
which needs b and all three components of r at plane z+1 (and r_z at z).
So a rank that owns the planes [z0, z1) of an nz-plane volume keeps an
extended volume of the planes [z0 - lo, z1 + hi), with lo = 1 unless
z0 = 0 and hi = 1 unless z1 = nz, and before every step

  * receives r_z of plane z0 - 1 from the rank below (one plane),
  * receives r_x, r_y, r_z of plane z1 from the rank above (three planes),
  * and, once per run, b of plane z1 from the rank above,

then runs one ordinary step on its extended volume.  The extended volume's
first and last planes are volume faces to the step, but only the halo planes
themselves see the difference (their z and their updates are wrong and are
never read): the owned planes come out exactly as on the whole volume.  The
exchange is point to point between neighbours, one plane up and three down
per step, 16 nx ny bytes; nothing is reduced.

The step and the momentum schedule are supplied by the caller: on GPUs the
library's tvfgp_step on a handle of the extended shape (``library_step``)
and tvfgp_momentum; the same host logic runs on the CPU with any other step
of the same signature.  Planes move with torch.distributed point-to-point
sends of contiguous plane tensors (NCCL between GPUs, gloo on the CPU), or,
for several slabs held by one process, with plain tensor copies
(``exchange_local``).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class SlabPlan:
    """The planes one rank owns and the halo planes around them."""
    rank: int
    world: int
    nz: int          # planes of the whole volume
    z0: int          # first owned plane
    z1: int          # one past the last owned plane
    lo: int          # halo planes below (0 or 1)
    hi: int          # halo planes above (0 or 1)

    @property
    def nz_ext(self) -> int:
        """Planes of the extended volume."""
        return self.z1 - self.z0 + self.lo + self.hi

    @property
    def owned(self) -> slice:
        """The owned planes as a slice of the extended volume's plane axis."""
        return slice(self.lo, self.lo + self.z1 - self.z0)


def partition(nz: int, world: int) -> list[SlabPlan]:
    """Split nz planes into `world` slabs as even as possible (the first
    nz % world slabs get one plane more).  Every rank owns at least one
    plane."""
    if world < 1 or nz < world:
        raise ValueError("need 1 <= world <= nz (got world %d, nz %d)" % (world, nz))
    base, extra = divmod(nz, world)
    plans, z = [], 0
    for rank in range(world):
        n = base + (1 if rank < extra else 0)
        plans.append(SlabPlan(rank, world, nz, z, z + n, 1 if z > 0 else 0, 1 if z + n < nz else 0))
        z += n
    return plans


def extend(plan: SlabPlan, whole):
    """The extended slab (planes [z0 - lo, z1 + hi)) of a whole volume,
    scalar (nz, ny, nx) or dual (3, nz, ny, nx), as a contiguous copy."""
    sl = slice(plan.z0 - plan.lo, plan.z1 + plan.hi)
    part = whole[..., sl, :, :]
    return part.contiguous() if hasattr(part, "contiguous") else part.copy()


# ---------------------------------------------------------------------------
# halo exchange
# ---------------------------------------------------------------------------

def exchange_dist(dist, plan: SlabPlan, r_ext, b_ext=None) -> None:
    """Fill the halo planes of this rank's r (and b, if given) from its
    neighbours with point-to-point sends: r_z of the plane below, all of r
    (and b) of the plane above.  Every rank of the group calls it.  The
    tensors are (3, nz_ext, ny, nx) and (nz_ext, ny, nx); a plane of one
    component is contiguous, so it is sent as it lies."""
    ops = []
    top = plan.lo + (plan.z1 - plan.z0) - 1          # last owned plane, extended index
    first = plan.lo                                  # first owned plane
    if plan.hi:                                      # neighbour above: rank + 1
        up = plan.rank + 1
        ops.append(dist.P2POp(dist.isend, r_ext[2, top], up))
        for a in range(3):
            ops.append(dist.P2POp(dist.irecv, r_ext[a, top + 1], up))
        if b_ext is not None:
            ops.append(dist.P2POp(dist.irecv, b_ext[top + 1], up))
    if plan.lo:                                      # neighbour below: rank - 1
        down = plan.rank - 1
        ops.append(dist.P2POp(dist.irecv, r_ext[2, 0], down))
        for a in range(3):
            ops.append(dist.P2POp(dist.isend, r_ext[a, first], down))
        if b_ext is not None:
            ops.append(dist.P2POp(dist.isend, b_ext[first], down))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()


def exchange_local(plans: list[SlabPlan], r_exts: list, b_exts: list | None = None) -> None:
    """The same exchange for slabs that one process holds (tensor copies)."""
    for k in range(len(plans) - 1):
        lo_p, hi_p = plans[k], plans[k + 1]
        top = lo_p.lo + (lo_p.z1 - lo_p.z0) - 1
        first = hi_p.lo
        r_exts[k + 1][2, 0].copy_(r_exts[k][2, top])
        r_exts[k][:, top + 1].copy_(r_exts[k + 1][:, first])
        if b_exts is not None:
            b_exts[k][top + 1].copy_(b_exts[k + 1][first])


# ---------------------------------------------------------------------------
# runs
# ---------------------------------------------------------------------------

def library_step(nx: int, ny: int, plan: SlabPlan, variant="auto"):
    """A step on the rank's extended volume through the CUDA library:
    returns (step, close) where step(b, p, r_src, r_dst, lam, m) enqueues
    tvfgp_step on the current stream."""
    from fgp_dual_stencil_gb300 import tvfgp as T
    h = T.Tvfgp(nx, ny, plan.nz_ext, variant)

    def step(b, p, r_src, r_dst, lam, m):
        h.step(b, p, r_src, r_dst, lam, m)

    return step, h.close


def library_schedule(t0: float, nsteps: int):
    """The momentum weights m_0..m_{n-1} and t after the last step, from the
    library's host code."""
    from fgp_dual_stencil_gb300 import tvfgp as T
    return T.tvfgp_momentum(t0, nsteps)


def run_slab(dist, plan: SlabPlan, step, schedule, b_ext, p_ext, r_ext, r_tmp, lam: float,
             nsteps: int, t0: float = 1.0) -> float:
    """nsteps FGP steps of the whole volume, of which this rank computes its
    slab.  b_ext, p_ext, r_ext hold the extended slab; r_tmp is a second
    buffer shaped like r_ext.  On return p_ext and r_ext hold the owned
    planes after the last step (halo planes are undefined).  b's upper halo
    is exchanged once here.  Returns t after the last step."""
    m, t_final = schedule(t0, nsteps)
    if nsteps == 0:
        return t_final
    src, dst = r_ext, r_tmp
    for k in range(nsteps):
        exchange_dist(dist, plan, src, b_ext if k == 0 else None)
        step(b_ext, p_ext, src, dst, lam, m[k])
        src, dst = dst, src
    if src is not r_ext:
        r_ext.copy_(src)
    return t_final


def run_local(plans: list[SlabPlan], steps: list, schedule, b_exts: list, p_exts: list, r_exts: list,
              r_tmps: list, lam: float, nsteps: int, t0: float = 1.0) -> float:
    """run_slab for every slab of one process, the exchange done by copies
    (each step's exchange completes before any slab's step starts)."""
    m, t_final = schedule(t0, nsteps)
    src, dst = list(r_exts), list(r_tmps)
    for k in range(nsteps):
        exchange_local(plans, src, b_exts if k == 0 else None)
        for j, step in enumerate(steps):
            step(b_exts[j], p_exts[j], src[j], dst[j], lam, m[k])
        src, dst = dst, src
    for j in range(len(plans)):
        if src[j] is not r_exts[j]:
            r_exts[j].copy_(src[j])
    return t_final
