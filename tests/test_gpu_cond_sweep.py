"""A seeded sweep of small random problems through the conditioning-token path
("Tiled Data Parallelism (TDP)", sections "Shared negative (reference) positions" and
"Position normalization"): bounds, filter (tdp_norm_filter, or the fused tdp_split_filter),
then the conditioning blend from the slots (tdp_cond_blend) and from per-block records
(tdp_cond_records + tdp_cond_blend_records).

Each draw picks the batch, grid, channels and dtype, the tiles and overlaps per dimension,
the number of conditioning tokens (some past 8192, where tdp_norm_filter takes its two-launch
form), the fraction with negative time, whether positions are normalised, and a row capacity
ncap at, below or far below the largest count.  The bounds and every filter output are
compared with the oracle exactly; the slot path's outputs with the fp64 oracle within the
blend tolerance; the records path's outputs bit for bit with the slot path's."""
import numpy as np
import pytest

import oracle
import workloads as wk
from gpu_path import assert_blend_close, assert_filter_equal, fill_sentinel, run_split_filter, to_dev, to_host

pytestmark = pytest.mark.gpu

CASES = 24


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


def _draw(tdp, rng):
    """A random problem the plan accepts, and its plan."""
    for _ in range(500):
        dtype = "bf16" if rng.random() < 0.7 else "f32"
        C = int(rng.choice([8, 16, 24, 40, 64, 136])) if dtype == "bf16" else int(rng.choice([4, 12, 20, 36]))
        B = int(rng.integers(1, 4))
        F, H, W = int(rng.integers(1, 7)), int(rng.integers(2, 41)), int(rng.integers(2, 49))
        n = (int(rng.integers(1, min(F, 3) + 1)), int(rng.integers(1, min(H, 9) + 1)),
             int(rng.integers(1, min(W, 9) + 1)))
        o = tuple(int(rng.integers(0, 4)) if n[d] > 1 else 0 for d in range(3))
        try:
            plan = tdp.tdp_plan_create(B, F, H, W, C, dtype, n, o)
        except tdp.TdpError:
            continue
        kind = rng.random()
        N = int(rng.integers(1, 64)) if kind < 0.3 else int(rng.integers(64, 2000)) if kind < 0.8 else \
            int(rng.integers(8193, 9000))
        neg = float(rng.choice([0.0, 0.05, 0.3]))
        wl = wk.Workload("sweep", B, F, H, W, C, dtype, n, o, N, neg, 0.05, int(rng.integers(1 << 30)))
        return wl, plan
    raise AssertionError("no valid problem drawn")


def _storage(wl, shape, rng):
    x = rng.standard_normal(shape, dtype=np.float32)
    return x if wl.dtype == "f32" else wk.f32_to_bf16_bits(x)


@pytest.mark.parametrize("case", range(CASES))
def test_cond_path_random_problem(tdp, case):
    import torch
    rng = np.random.default_rng(90210 + case)
    wl, plan = _draw(tdp, rng)
    normalize = bool(rng.random() < 0.8)
    fused = case % 2 == 1
    X, P, K = wk.make_inputs(wl)
    N = K.shape[2]
    out = run_split_filter(tdp, plan, wl, X, P, K, normalize=normalize, fused=fused)

    # bounds and filter against the oracle, exactly
    p = oracle.problem_of(wl)
    _, Q = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Q)
    assert np.array_equal(out["mn"], mn) and np.array_equal(out["mx"], mx)
    keep, idx, count, kcount, Kout, slot = oracle.filter_cond(p, K, mn, mx, normalize, with_slot=True)
    ref = dict(keep=keep, idx=idx, count=count, kcount=kcount, Kout=Kout, slot=slot)
    assert_filter_equal(out, ref, plan.n_tiles, wl.B)

    # the conditioning blend, at a row capacity at, below or far below the largest count
    top = max(1, int(count.max()))
    ncap = int(rng.choice([top, max(1, top // 2), 1]))
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    Yc = _storage(wl, (plan.n_tiles, wl.B, ncap, wl.C), rng)
    Ycd = to_dev(Yc)
    O1 = fill_sentinel(torch.empty((wl.B, N, wl.C), dtype=dt, device="cuda"))
    tdp.tdp_cond_blend(plan, N, ncap, Ycd, out["slotd"], O1)
    torch.cuda.synchronize()
    assert_blend_close(to_host(O1), oracle.cond_blend(p, Yc, keep, idx, count, ncap), wl)

    recs = torch.full((tdp.tdp_cond_records_size(plan, N),), -7, dtype=torch.int32, device="cuda")
    tdp.tdp_cond_records(plan, N, ncap, out["slotd"], recs)
    O2 = fill_sentinel(torch.empty_like(O1))
    tdp.tdp_cond_blend_records(plan, N, recs, Ycd, ncap, O2)
    torch.cuda.synchronize()
    assert torch.equal(O1.view(torch.uint8), O2.view(torch.uint8)), "records path differs from the slot path"
