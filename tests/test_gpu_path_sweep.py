"""A seeded sweep of small random problems through the whole hot path ("Tiled Data
Parallelism (TDP)", sections "What it is", "Position normalization" and "Shared negative
(reference) positions").

Each draw picks the batch, grid, channels and dtype, the tiles and overlaps per dimension
(uneven cores and overlaps up to the core size included), the number of conditioning tokens
(none in some draws) and whether positions are normalised.  Per draw:
- both forms of the pre-model stage (three calls, and tdp_split_filter) against the oracle
  bit for bit, the blend of noisy tile outputs within the blend tolerance of the fp64
  oracle, and the reconstruction property (test_gpu_parity's checks);
- tdp_split_tma against the oracle's split, bit for bit;
- tdp_blend_cond (blend and conditioning blend in one launch) against tdp_blend and
  tdp_cond_blend, bit for bit."""
import numpy as np
import pytest

import oracle
import workloads as wk
from gpu_path import fill_sentinel, run_split_filter, to_dev, to_host
from test_gpu_parity import _check_path, _yout

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
        B = int(rng.integers(1, 3))
        F, H, W = int(rng.integers(1, 9)), int(rng.integers(2, 41)), int(rng.integers(2, 49))
        n = (int(rng.integers(1, min(F, 3) + 1)), int(rng.integers(1, min(H, 9) + 1)),
             int(rng.integers(1, min(W, 9) + 1)))
        o = tuple(int(rng.integers(0, 6)) if n[d] > 1 else 0 for d in range(3))
        try:
            plan = tdp.tdp_plan_create(B, F, H, W, C, dtype, n, o)
        except tdp.TdpError:
            continue
        N = 0 if rng.random() < 0.15 else int(rng.integers(1, 1500))
        neg = float(rng.choice([0.0, 0.05, 0.3]))
        wl = wk.Workload("sweep", B, F, H, W, C, dtype, n, o, N, neg, 0.05, int(rng.integers(1 << 30)))
        return wl, plan
    raise AssertionError("no valid problem drawn")


@pytest.mark.parametrize("case", range(CASES))
def test_path_random_problem(tdp, case):
    import torch
    rng = np.random.default_rng(31337 + case)
    wl, plan = _draw(tdp, rng)
    normalize = bool(rng.random() < 0.8)
    X, P, K = wk.make_inputs(wl)
    _check_path(tdp, wl, X, P, K, normalize=normalize)

    # the bulk-tensor split
    p = oracle.problem_of(wl)
    Yref, Qref = oracle.split(p, X, P)
    mn, _ = oracle.bounds(p, Qref)
    Qexp = oracle.normalize(p, Qref, mn) if normalize else Qref
    Y, Q, _, _ = tdp.alloc_split_outputs(plan, "cuda")
    for t in (Y, Q):
        fill_sentinel(t)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tdp.tdp_split_tma(plan, to_dev(X), to_dev(P), to_dev(mn), int(normalize), Y, Q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(to_host(Y).reshape(Yref.shape), Yref)
    assert np.array_equal(to_host(Q), Qexp)

    # the post-model stage in one launch against the two calls
    out = run_split_filter(tdp, plan, wl, X, P, K, normalize=normalize, fused=True)
    N = K.shape[2]
    ncap = max(1, int(out["count"].max()) if out["count"].size else 1)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    Yout = to_dev(_yout(wl, Yref, wl.seed + 7))
    yc = rng.standard_normal((plan.n_tiles, wl.B, ncap, wl.C), dtype=np.float32)
    Ycd = to_dev(yc if wl.dtype == "f32" else wk.f32_to_bf16_bits(yc))
    Z1 = fill_sentinel(torch.empty((wl.B, wl.F, wl.H, wl.W, wl.C), dtype=dt, device="cuda"))
    O1 = fill_sentinel(torch.empty((wl.B, N, wl.C), dtype=dt, device="cuda"))
    tdp.tdp_blend(plan, Yout, Z1)
    tdp.tdp_cond_blend(plan, N, ncap, Ycd, out["slotd"], O1)
    Z2, O2 = fill_sentinel(torch.empty_like(Z1)), fill_sentinel(torch.empty_like(O1))
    tdp.tdp_blend_cond(plan, Yout, Z2, N, ncap, Ycd, out["slotd"], O2)
    torch.cuda.synchronize()
    assert torch.equal(Z1.view(torch.uint8), Z2.view(torch.uint8))
    assert torch.equal(O1.view(torch.uint8), O2.view(torch.uint8))
