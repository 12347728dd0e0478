"""The run planner, on the host (no GPU): for every shape class, row pitch,
variant and step count, the launches tvfgp_run would enqueue must take p and
r from the caller's buffers back to them, never read a buffer they write in
the same launch, apply the momentum weights of the schedule in order, and
use the packing and padded-output launches exactly where the header says;
and the two-step kernel's split of the planes among its CTAs must cover
every plane once."""
import itertools

import numpy as np
import pytest

from fgp_dual_stencil_gb300 import tvfgp as T

B, P, R, SCRATCH = 0, 1, 2, 3
PACKED_B, PACKED_P, PACKED_R, SHADOW_SCRATCH = 7, 8, 9, 10
TWO, PACK, PADDED_OUT, HALF = 1, 2, 4, 8

SHAPES = [(64, 16, 16, 0), (33, 5, 7, 0), (62, 8, 8, 0), (64, 16, 16, 66), (64, 16, 16, 67),
          (62, 8, 8, 64), (33, 5, 7, 34), (8, 4, 3, 0), (8, 4, 3, 10)]


def expected_route(nx, pitch, variant, n):
    padded = pitch not in (0, nx)
    if not padded or nx % 4 or n < 4 or variant not in ("auto", "zmarch", "zmarch2", "cube"):
        return 0
    if variant in ("auto", "zmarch2") and pitch % 2 == 0:
        return 1
    return 2


def replay(route, copy_back, launches):
    """Follow p and r through the launches; returns (p, r, steps, weights)."""
    p, r = (PACKED_P, PACKED_R) if route == 2 else (P, R)
    steps, weights = 0, []
    k = 0
    while k < len(launches):
        L = launches[k]
        roles = (L["b"], L["p_src"], L["p_dst"], L["r_src"], L["r_dst"])
        assert min(roles) >= 0, L
        assert L["p_src"] == p and L["r_src"] == r, (L, p, r)
        assert L["r_dst"] != L["r_src"] and L["r_dst"] not in (L["p_src"], L["p_dst"]), L
        if L["flags"] & HALF:
            # the two kernels of one step: z from r_src, then the rest
            M = launches[k + 1]
            assert M["flags"] & HALF and (M["r_src"], M["r_dst"], M["m"]) == (L["r_src"], L["r_dst"], L["m"])
            assert L["p_dst"] == L["p_src"] == M["p_src"] == M["p_dst"]
            steps += 1
            weights.append(L["m"][0])
            r = L["r_dst"]
            k += 2
            continue
        if L["flags"] & TWO:
            assert L["p_dst"] != L["p_src"], L
            assert len({L["p_src"], L["p_dst"], L["r_src"], L["r_dst"]}) == 4, L
            steps += 2
            weights += list(L["m"])
        else:
            if not L["flags"] & PACK:
                assert L["p_dst"] == L["p_src"], L            # one step updates p in place
            steps += 1
            weights.append(L["m"][0])
        p, r = L["p_dst"], L["r_dst"]
        k += 1
    if copy_back:
        assert r == (SHADOW_SCRATCH if route == 2 else SCRATCH)
        r = PACKED_R if route == 2 else R
    return p, r, steps, weights


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("variant", sorted(T.VARIANTS))
def test_plans_route_the_dual_home_in_schedule_order(shape, variant):
    nx, ny, nz, pitch = shape
    for n, t0 in itertools.product(range(0, 12), (1.0, 2.5)):
        route, copy_back, launches = T.tvfgp_debug_plan(nx, ny, nz, pitch, variant, n, t0)
        assert route == expected_route(nx, pitch, variant, n), (shape, variant, n)
        if n == 0:
            assert launches == [] and not copy_back
            continue
        p, r, steps, weights = replay(route, copy_back, launches)
        home = (PACKED_P, PACKED_R) if route == 2 else (P, R)
        assert (p, r) == home, (shape, variant, n, route)
        assert steps == n
        m, _ = T.tvfgp_momentum(t0, n)
        assert np.array_equal(np.float32(weights), np.float32(m)), (shape, variant, n)
        flags = [L["flags"] for L in launches]
        bs = [L["b"] for L in launches]
        if route == 1:
            assert flags[0] == PACK and flags[-1] == TWO | PADDED_OUT
            assert not any(f & (PACK | PADDED_OUT) for f in flags[1:-1])
            assert bs[0] == B and set(bs[1:]) == {PACKED_B}
            assert not copy_back
        else:
            assert not any(f & (PACK | PADDED_OUT) for f in flags)
            assert set(bs) == {PACKED_B if route == 2 else B}
        # the two-step kernel is used from four steps on wherever it can run
        two = [L for L in launches if L["flags"] & TWO]
        dense4 = pitch in (0, nx) and nx % 4 == 0
        if variant in ("auto", "zmarch2") and n >= 4 and (dense4 or route):
            assert len(two) == (n - 1) // 2 if route == 1 else len(two) == n // 2
        else:
            assert not two or route == 2


def test_plan_argument_checks():
    for args in [(0, 4, 4, 0, "auto", 1), (8, 4, 4, 7, "auto", 1), (8, 4, 4, 0, "auto", -1),
                 (65535, 65535, 1, 0, "auto", 1)]:
        with pytest.raises(T.TvfgpError):
            T.tvfgp_debug_plan(*args)


def test_two_step_chunks_partition_the_planes():
    """The two-step kernel's split of the planes among its CTAs covers every
    plane once, no chunk is empty or longer than zc, and the last chunk is
    cut into three pieces exactly when the last round of CTAs over the
    resident slots is less than half full."""
    cand = (128, 96, 64, 48, 32, 24, 16, 12, 8)
    for nx, ny in [(512, 512), (1000, 600), (256, 256), (64, 26), (33, 5), (2048, 1024)]:
        tiles = -(-nx // 32) * -(-ny // 12)
        for nz in list(range(1, 70)) + [127, 128, 129, 255, 256, 257, 300, 511, 512, 513, 1100]:
            for slots in (1, 152, 304, 456, 608):
                zc, chunks = T.tvfgp_debug_chunks(nx, ny, nz, slots)
                assert zc in cand
                assert [z for a, b in chunks for z in range(a, b)] == list(range(nz)), (nx, ny, nz, slots)
                assert all(0 < b - a <= zc for a, b in chunks)
                whole = -(-nz // zc)
                last = nz - (whole - 1) * zc
                rem = tiles * whole % slots
                tapered = len(chunks) != whole
                assert tapered == (whole > 1 and last >= 24 and rem * 2 < slots), (nx, ny, nz, slots)
                if tapered:
                    sizes = [b - a for a, b in chunks[-3:]]
                    assert len(chunks) == whole + 2 and sum(sizes) == last and sizes[0] >= sizes[1] >= sizes[2]
    with pytest.raises(T.TvfgpError):
        T.tvfgp_debug_chunks(8, 8, 8, 0)
