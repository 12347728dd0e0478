"""z-slab decomposition of the FGP step (fgp_dual_stencil_gb300/slabs.py).

On the CPU: the partition and halo layout, and 2 and 3 gloo ranks that each
run the oracle's step on their extended slab, exchanging halo planes with
torch.distributed point-to-point sends; the owned planes, put together,
must equal the oracle's run on the whole volume bit for bit.  On one GPU:
three slabs held by one process, stepped by the library's tvfgp_step with
the exchange done by copies, against the same oracle run."""
import os
import socket
import sys

import numpy as np
import pytest

import oracle
from fgp_dual_stencil_gb300 import slabs, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("nz,world", [(1, 1), (7, 1), (7, 2), (7, 3), (10, 4), (5, 5), (300, 8)])
def test_partition_covers_every_plane_once(nz, world):
    plans = slabs.partition(nz, world)
    assert [p.rank for p in plans] == list(range(world))
    assert plans[0].z0 == 0 and plans[-1].z1 == nz
    for a, b in zip(plans, plans[1:]):
        assert a.z1 == b.z0
    sizes = [p.z1 - p.z0 for p in plans]
    assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    for p in plans:
        assert p.lo == (1 if p.z0 > 0 else 0) and p.hi == (1 if p.z1 < nz else 0)
        assert p.nz_ext == p.z1 - p.z0 + p.lo + p.hi
        assert p.owned.stop - p.owned.start == p.z1 - p.z0


def test_partition_rejects_more_ranks_than_planes():
    with pytest.raises(ValueError):
        slabs.partition(3, 4)
    with pytest.raises(ValueError):
        slabs.partition(3, 0)


def test_extend_takes_the_halo_planes():
    import torch
    vol = torch.arange(2 * 3 * 9, dtype=torch.float32).reshape(9, 3, 2)
    dual = torch.stack([vol, -vol, 2 * vol])
    for p in slabs.partition(9, 3):
        e = slabs.extend(p, vol)
        assert torch.equal(e, vol[p.z0 - p.lo:p.z1 + p.hi]) and e.is_contiguous()
        d = slabs.extend(p, dual)
        assert d.shape == (3, p.nz_ext, 3, 2) and torch.equal(d[:, p.owned], dual[:, p.z0:p.z1])


def oracle_step(b, p, r_src, r_dst, lam, m):
    """tvfgp_step's contract on CPU tensors, computed by the oracle."""
    pn = p.numpy()
    rd, _ = oracle.fgp_step(b.numpy(), pn, r_src.numpy(), np.float32(lam), np.float32(m))
    r_dst.copy_(__import__("torch").from_numpy(rd))


def case(shape, seed):
    b = synth.random_case(shape, seed)
    p0 = synth.random_dual(shape, seed + 1, scale=0.4)
    r0 = synth.random_dual(shape, seed + 2, scale=0.6)
    return b, p0, r0


def _rank_main(rank, world, port, shape, seed, lam, nsteps, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group(backend="gloo", rank=rank, world_size=world)
    b, p0, r0 = case(shape, seed)
    plan = slabs.partition(shape[2], world)[rank]
    tb, tp, tr = (torch.from_numpy(x) for x in (b, p0, r0))
    b_ext, p_ext, r_ext = slabs.extend(plan, tb), slabs.extend(plan, tp), slabs.extend(plan, tr)
    # the halo planes start with nothing useful in them: the exchange fills
    # what the step reads
    b_ext[:plan.lo] = 0
    b_ext[b_ext.shape[0] - plan.hi:] = 0
    r_ext[:, :plan.lo] = float("nan")
    r_ext[:, r_ext.shape[1] - plan.hi:] = float("nan")
    r_tmp = torch.empty_like(r_ext)
    t = slabs.run_slab(dist, plan, oracle_step, oracle.momentum, b_ext, p_ext, r_ext, r_tmp, lam, nsteps, 1.0)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, plan.z0, plan.z1, p_ext[:, plan.owned].numpy().copy(), r_ext[:, plan.owned].numpy().copy(), t))


@pytest.mark.parametrize("world,shape,nsteps", [(2, (12, 9, 10), 6), (3, (9, 7, 8), 5), (3, (8, 5, 3), 4)])
def test_gloo_slabs_equal_the_whole_volume(world, shape, nsteps):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    lam, seed = 0.05, 61
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, shape, seed, lam, nsteps, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    b, p0, r0 = case(shape, seed)
    po, ro = p0.copy(), r0.copy()
    t_whole = oracle.fgp_run(b, po, ro, lam, nsteps, 1.0)
    for rank, z0, z1, ps, rs, t in res:
        assert t == t_whole
        assert np.array_equal(ps, po[:, z0:z1]), "rank %d: p differs" % rank
        assert np.array_equal(rs, ro[:, z0:z1]), "rank %d: r differs" % rank
    assert [(z0, z1) for _, z0, z1, *_ in res][-1][1] == shape[2]


@pytest.mark.gpu
@pytest.mark.parametrize("shape,parts,nsteps", [((64, 40, 30), 3, 7), ((36, 20, 9), 4, 4)])
def test_library_slabs_on_one_gpu_equal_the_oracle(shape, parts, nsteps):
    import torch
    from fgp_dual_stencil_gb300 import tvfgp as T
    assert torch.cuda.is_available()
    nx, ny, nz = shape
    lam = 0.05
    b, p0, r0 = case(shape, 81)
    plans = slabs.partition(nz, parts)
    tb, tp, tr = (torch.from_numpy(x).cuda() for x in (b, p0, r0))
    b_exts = [slabs.extend(p, tb) for p in plans]
    p_exts = [slabs.extend(p, tp) for p in plans]
    r_exts = [slabs.extend(p, tr) for p in plans]
    r_tmps = [torch.empty_like(r) for r in r_exts]
    made = [slabs.library_step(nx, ny, p) for p in plans]
    try:
        t = slabs.run_local(plans, [s for s, _ in made], slabs.library_schedule, b_exts, p_exts, r_exts,
                            r_tmps, lam, nsteps, 1.0)
        torch.cuda.synchronize()
    finally:
        for _, close in made:
            close()
    po, ro = p0.copy(), r0.copy()
    t_whole = oracle.fgp_run(b, po, ro, lam, nsteps, 1.0)
    assert t == t_whole
    for p, pe, re in zip(plans, p_exts, r_exts):
        assert np.array_equal(pe[:, p.owned].cpu().numpy(), po[:, p.z0:p.z1])
        assert np.array_equal(re[:, p.owned].cpu().numpy(), ro[:, p.z0:p.z1])
