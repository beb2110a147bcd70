"""GPU parity of the two reductions over tiles besides the latent blend, against the
CPU oracle: each conditioning token's outputs averaged over the tiles that kept it
("Tiled Data Parallelism (TDP)", "Shared negative (reference) positions": weight
1/(tiles that kept it)), and the audio mean over tiles ("What it is")."""
import numpy as np
import pytest

import oracle
import workloads as wk
from gpu_path import as_f64, assert_blend_close, run_split_filter, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


def _plan(tdp, wl):
    return tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)


def _random_storage(wl, shape, seed):
    x = np.random.default_rng(seed).standard_normal(shape, dtype=np.float32)
    return x if wl.dtype == "f32" else wk.f32_to_bf16_bits(x)


def _cond_case(tdp, wl, ncap=None, seed=0):
    import torch
    X, P, K = wk.make_inputs(wl)
    plan = _plan(tdp, wl)
    p = oracle.problem_of(wl)
    out = run_split_filter(tdp, plan, wl, X, P, K)
    N = K.shape[2]
    ncap = max(1, int(out["count"].max())) if ncap is None else ncap
    Yc = _random_storage(wl, (plan.n_tiles, wl.B, ncap, wl.C), seed)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    res = torch.full((wl.B, N, wl.C), float("nan"), dtype=dt, device="cuda")
    tdp.tdp_cond_blend(plan, N, ncap, to_dev(Yc), out["slotd"], res)
    torch.cuda.synchronize()
    ref = oracle.cond_blend(p, Yc, out["keep"], out["idx"], out["count"], ncap)
    got = to_host(res)
    assert_blend_close(got, ref, wl)
    return out, got, ref


@pytest.mark.parametrize("name", ["tiny", "small", "medium", "temporal"])
def test_cond_blend_parity(tdp, name):
    out, got, ref = _cond_case(tdp, wk.by_name(name))
    unkept = out["kcount"] == 0
    assert (as_f64(got)[unkept] == 0).all()


def test_cond_blend_truncated_rows(tdp):
    """Rows reserved per (tile, batch) below the largest count: later kept tokens are
    ignored on both sides."""
    _cond_case(tdp, wk.by_name("small"), ncap=7)


def test_cond_blend_one_row_per_tile(tdp):
    """One row reserved per (tile, batch item): only each tile's first kept token is
    stored, so most blocks of 8 tokens hold no stored row at all (their outputs are all
    zero) while their tokens still carry the full 1/kcount weight."""
    out, got, ref = _cond_case(tdp, wk.by_name("small").replace(B=2), ncap=1)
    stored = (out["slot"] == 0).any(axis=0)                   # [B, N]: some tile stored the token
    assert (~stored).sum() > 0.9 * stored.size
    assert (as_f64(got)[~stored] == 0).all()


def test_cond_blend_large_workload(tdp):
    _cond_case(tdp, wk.by_name("large"))


@pytest.mark.parametrize("name,L", [("tiny", 20), ("small", 4096), ("temporal", 2048 * 8 + 8)])
def test_tile_mean_parity(tdp, name, L):
    import torch
    wl = wk.by_name(name)
    plan = _plan(tdp, wl)
    A = _random_storage(wl, (plan.n_tiles, wl.B, L), 3)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    res = torch.full((wl.B, L), float("nan"), dtype=dt, device="cuda")
    tdp.tdp_tile_mean(plan, L, to_dev(A), res)
    torch.cuda.synchronize()
    assert_blend_close(to_host(res), oracle.tile_mean(oracle.problem_of(wl), A, L), wl)


def test_reductions_empty(tdp):
    import torch
    wl = wk.by_name("small")
    plan = _plan(tdp, wl)
    e = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    tdp.tdp_cond_blend(plan, 0, 1, torch.empty(plan.n_tiles * wl.B * wl.C, dtype=torch.bfloat16, device="cuda"),
                       torch.empty(0, dtype=torch.int32, device="cuda"), e)
    tdp.tdp_tile_mean(plan, 0, e, e)
    torch.cuda.synchronize()


def test_cond_blend_many_tiles(tdp):
    wl = wk.by_name("tiny").replace(F=4, H=64, W=64, C=8, dtype="bf16", num_tiles=(2, 32, 32),
                                    overlap=(1, 2, 1), n_cond=300)
    _cond_case(tdp, wl)


def test_cond_blend_ragged_tokens(tdp):
    """A token count that is not a multiple of 8, 16 or 32 (the last block of tokens of each
    batch item is part-filled), two batch items."""
    _cond_case(tdp, wk.by_name("small").replace(B=2, n_cond=1003))


def test_cond_blend_wide_channels(tdp):
    """4 KB rows (bf16 C=2048): 256 vectors per token, sixteen slabs of 16 lanes."""
    wl = wk.by_name("tiny").replace(F=2, H=6, W=10, C=2048, dtype="bf16", num_tiles=(1, 2, 2),
                                    overlap=(0, 2, 2), n_cond=100)
    _cond_case(tdp, wl)


@pytest.mark.parametrize("nw", [16, 17])
def test_cond_blend_tile_count_edges(tdp, nw):
    """256 tiles (the largest count the row kernel takes) and 272 (the warp-per-token kernel)."""
    wl = wk.by_name("tiny").replace(F=2, H=48, W=52, C=8, dtype="bf16", num_tiles=(1, 16, nw),
                                    overlap=(0, 1, 1), n_cond=200)
    _cond_case(tdp, wl)


def test_cond_blend_rows_across_stages(tdp):
    """256 tiles and 1 KB rows (bf16 C=512: 64 vectors, four slabs of 16 lanes): a token
    kept by every tile has 256 rows, more than five stages of the row ring, so its sum
    continues from stage to stage and from slab to slab; half the tokens have negative
    time."""
    wl = wk.by_name("tiny").replace(F=2, H=48, W=52, C=512, dtype="bf16", num_tiles=(1, 16, 16),
                                    overlap=(0, 1, 1), n_cond=120, neg_frac=0.5)
    out, _, _ = _cond_case(tdp, wl)
    assert int(out["kcount"].max()) == 256


def test_cond_blend_odd_vector_count(tdp):
    """bf16 C=136: 17 channel vectors, two slabs, the second with one vector (15 of a
    token's 16 lanes idle)."""
    wl = wk.by_name("tiny").replace(F=4, H=24, W=40, C=136, dtype="bf16", num_tiles=(2, 4, 8),
                                    overlap=(1, 2, 2), n_cond=400)
    _cond_case(tdp, wl)
