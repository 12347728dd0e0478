"""A volume past 2^31 voxels: 2048 x 1024 x 1100 (9.2 GB per volume), where
plane z = 1024 starts at voxel 2^31 and a 32-bit voxel index would wrap.

The volume is far too large for the oracle, so each kernel is checked on
sub-boxes.  One FGP step at voxel i reads r and p only at offsets with
components in {-1, 0, 1} (z at i and i + e_a, each from r at j and j - e_c),
so after k steps a voxel depends only on the inputs within k voxels of it
(L-infinity), and the primal of the result on one voxel more.  The oracle
run on a box, with the box's own faces as volume faces, therefore gives the
exact result on every voxel farther than that from the faces of the box
that are not faces of the volume.  The inputs come from torch's seeded
generator on the device; the boxes of them that the oracle reads are copied
to the host before the run."""
import numpy as np
import pytest

import oracle

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

NX, NY, NZ = 2048, 1024, 1100
LAM = 0.05


def boxes():
    """(x0, x1, y0, y1, z0, z1): the first planes, the planes around voxel
    2^31 (plane 1024), the last planes and a corner of every upper face."""
    return [(0, 40, 0, 24, 0, 12),
            (NX // 2 - 20, NX // 2 + 20, NY // 2 - 12, NY // 2 + 12, 1016, 1032),
            (NX - 40, NX, NY - 24, NY, NZ - 12, NZ)]


def inner(box, margin):
    """Slices, in box coordinates, of the voxels farther than `margin` from
    every face of the box that is not a face of the volume."""
    x0, x1, y0, y1, z0, z1 = box
    out = []
    for lo, hi, n in ((z0, z1, NZ), (y0, y1, NY), (x0, x1, NX)):
        a = 0 if lo == 0 else margin
        b = hi - lo if hi == n else hi - lo - margin
        assert b > a
        out.append(slice(a, b))
    return tuple(out)


def take(t, box):
    x0, x1, y0, y1, z0, z1 = box
    return np.ascontiguousarray(t[..., z0:z1, y0:y1, x0:x1].cpu().numpy())


@pytest.fixture(scope="module")
def volumes():
    import torch
    if torch.cuda.get_device_properties(0).total_memory < 200 * 2**30:
        pytest.skip("needs about 190 GB of device memory")
    g = torch.Generator(device="cuda")
    b = torch.empty((NZ, NY, NX), device="cuda")
    p = torch.empty((3, NZ, NY, NX), device="cuda")
    r = torch.empty_like(p)
    z = torch.empty_like(b)

    def reset():
        g.manual_seed(20261202)
        torch.rand(b.shape, generator=g, device="cuda", out=b)
        torch.rand(p.shape, generator=g, device="cuda", out=p)
        p.sub_(0.5).mul_(0.8)
        torch.rand(r.shape, generator=g, device="cuda", out=r)
        r.sub_(0.5).mul_(1.2)

    reset()
    start = [(take(b, bx), take(p, bx), take(r, bx)) for bx in boxes()]
    yield b, p, r, z, reset, start
    del b, p, r, z
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant,nsteps", [("auto", 5), ("zmarch", 3), ("fused", 3), ("scalar", 2),
                                            ("cube", 2), ("separate", 2)])
def test_past_2_31_voxels_matches_the_oracle_on_boxes(volumes, variant, nsteps):
    import torch
    from fgp_dual_stencil_gb300 import tvfgp as T
    b, p, r, z, reset, start = volumes
    reset()
    with T.Tvfgp(NX, NY, NZ, variant) as h:
        h.run(b, p, r, LAM, nsteps, 1.0)
        h.primal(b, p, LAM, z=z)
        assert h.check() == 0
    torch.cuda.synchronize()
    for bx, (b0, p0, r0) in zip(boxes(), start):
        po, ro = p0.copy(), r0.copy()
        oracle.fgp_run(b0, po, ro, LAM, nsteps, 1.0)
        zo = oracle.primal(b0, po, LAM)
        s = inner(bx, nsteps)
        assert np.array_equal(take(p, bx)[(slice(None),) + s], po[(slice(None),) + s]), (variant, bx, "p")
        assert np.array_equal(take(r, bx)[(slice(None),) + s], ro[(slice(None),) + s]), (variant, bx, "r")
        s1 = inner(bx, nsteps + 1)
        assert np.array_equal(take(z, bx)[s1], zo[s1]), (variant, bx, "z")
