"""Host-only plan helpers: balanced h x w grid for a world size, tile count for a
largest tile size, and the round-robin tile-to-rank assignment ("Tiled Data
Parallelism (TDP)", sections "What it is" and "API")."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


def test_balanced_tile_split_is_the_squarest_factorisation(tdp):
    for world in range(1, 257):
        h, w = tdp.tdp_balanced_tile_split(world)
        assert h * w == world and 1 <= h <= w
        pairs = [(a, world // a) for a in range(1, world + 1) if world % a == 0]
        assert w - h == min(abs(b - a) for a, b in pairs)
    assert tdp.tdp_balanced_tile_split(4) == (2, 2)
    assert tdp.tdp_balanced_tile_split(8) == (2, 4)
    with pytest.raises(tdp.TdpError):
        tdp.tdp_balanced_tile_split(0)


def test_round_robin_golden(tdp):
    with open(os.path.join(GOLDEN, "round_robin.txt")) as fh:
        nt, world, per = (int(x) for x in [l for l in fh if not l.startswith("#")][0].split())
    plan = tdp.tdp_plan_create(1, 16, 16, 16, 8, "bf16", (1, 4, 4), (0, 2, 2))
    assert plan.n_tiles == nt
    for r in range(world):
        assert len(tdp.tdp_rank_tiles(plan, r, world)) == per


def test_round_robin_partition(tdp):
    plan = tdp.tdp_plan_create(1, 64, 128, 192, 8, "bf16", (2, 8, 8), (4, 16, 16))
    for world in (1, 3, 7, 8, 128, 200):
        owned = [tdp.tdp_rank_tiles(plan, r, world) for r in range(world)]
        allt = np.sort(np.concatenate(owned))
        assert np.array_equal(allt, np.arange(plan.n_tiles))
        sizes = [len(o) for o in owned]
        assert max(sizes) - min(sizes) <= 1
        for r, o in enumerate(owned):
            assert (o % world == r).all() and np.all(np.diff(o) > 0)
    with pytest.raises(tdp.TdpError):
        tdp.tdp_rank_tiles(plan, 3, 3)


def test_tiles_for_size_is_the_smallest_fitting_count(tdp):
    for L in (1, 7, 20, 64, 128, 192):
        for o in (0, 1, 2, 5, 8, 16):
            for size in (1, 3, 8, 16, 24, 40, 64, 200):
                sizes = {}
                for n in range(1, min(L, 64) + 1):
                    try:
                        lo, hi = oracle.tile_boxes_1d(L, n, o)
                    except ValueError:
                        continue
                    sizes[n] = int((hi - lo).max())
                fit = [n for n, m in sizes.items() if m <= size]
                if fit:
                    assert tdp.tdp_tiles_for_size(L, size, o) == min(fit)
                else:
                    with pytest.raises(tdp.TdpError):
                        tdp.tdp_tiles_for_size(L, size, o)
