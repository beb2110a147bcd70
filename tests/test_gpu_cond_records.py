"""tdp_cond_records + tdp_cond_blend_records, the conditioning-token output reduction in two
calls ("Tiled Data Parallelism (TDP)", "Shared negative (reference) positions": weight
1/(tiles that kept it)): the outputs are bit for bit those of tdp_cond_blend, which the
reduction tests compare with the CPU oracle; the records themselves, and the deal of the
tokens to them, are checked against the filter's slots and counts."""
import numpy as np
import pytest

import oracle
import workloads as wk
from gpu_path import assert_blend_close, fill_sentinel, run_split_filter, to_dev, to_host

pytestmark = pytest.mark.gpu

TOK = 8          # tokens per block
HEAD = 2 + 3 * TOK
CLASSES = 16     # classes of stored rows the deal ranks tokens by


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


def _storage(wl, shape, seed):
    x = np.random.default_rng(seed).standard_normal(shape, dtype=np.float32)
    return x if wl.dtype == "f32" else wk.f32_to_bf16_bits(x)


def _setup(tdp, wl, ncap=None):
    X, P, K = wk.make_inputs(wl)
    plan = tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)
    out = run_split_filter(tdp, plan, wl, X, P, K, fused=True)
    N = K.shape[2]
    ncap = max(1, int(out["count"].max())) if ncap is None else ncap
    return plan, out, N, ncap


def _blends(tdp, plan, wl, out, N, ncap, seeds=(11,)):
    import torch
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    n = tdp.tdp_cond_records_size(plan, N)
    recs = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    tdp.tdp_cond_records(plan, N, ncap, out["slotd"], recs)
    res = []
    for seed in seeds:
        Yc = to_dev(_storage(wl, (plan.n_tiles, wl.B, ncap, wl.C), seed))
        O1 = fill_sentinel(torch.empty((wl.B, N, wl.C), dtype=dt, device="cuda"))
        O2 = fill_sentinel(torch.empty((wl.B, N, wl.C), dtype=dt, device="cuda"))
        tdp.tdp_cond_blend(plan, N, ncap, Yc, out["slotd"], O1)
        tdp.tdp_cond_blend_records(plan, N, recs, Yc, ncap, O2)
        torch.cuda.synchronize()
        res.append((Yc, O1, O2))
    return recs, res


def _same(a, b):
    import torch
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def _check_records(plan, wl, out, N, ncap, recs):
    """The deal: tokens ranked by class min(rows // width, 15) of their stored rows, classes in
    descending order and tokens of a class in ascending order, rank r at place r // G of record
    r % G (rounds alternate direction); every token once.  Every token's info (tiles that kept
    it, stored rows) and, on a sample, its list.  Record i: its tokens, their stored rows in
    ascending tile order, the rows per token and the tiles that kept each token."""
    B, nt = wl.B, plan.n_tiles
    G = B * ((N + TOK - 1) // TOK)
    stride = (HEAD + TOK * nt + 3) // 4 * 4
    r = recs.cpu().numpy()
    slot = out["slot"]                                     # [nt, B, N]
    kcount = out["kcount"]                                 # [B, N]
    stored = (slot >= 0) & (slot < ncap)
    lens = stored.sum(0).reshape(-1)                       # token b N + k
    width = (nt + CLASSES) // CLASSES
    cls = np.minimum(lens // width, CLASSES - 1)
    order = np.argsort(-cls, kind="stable")
    want = np.full((G, TOK), -1, np.int64)
    for rank, tok in enumerate(order):
        q, p = divmod(rank, G)
        want[G - 1 - p if q % 2 else p, q] = tok
    assign = r[G * stride:G * stride + G * TOK].reshape(G, TOK)
    assert np.array_equal(assign, want), "the deal differs"
    info = r[G * stride + G * TOK:G * stride + G * TOK + B * N]
    assert np.array_equal(info & 0xffff, lens) and np.array_equal(info >> 16, kcount.reshape(-1))
    lists = r[G * stride + 2 * G * TOK:].view(np.uint32)
    for tok in range(0, B * N, max(1, B * N // 64)):
        b, k = divmod(tok, N)
        mine = [(t * B + b) * ncap + slot[t, b, k] for t in range(nt) if stored[t, b, k]]
        assert lists[tok * nt:tok * nt + len(mine)].tolist() == mine
    for i in range(G):
        rec = r[i * stride:(i + 1) * stride]
        assert rec[0] == i
        rows = []
        for j in range(TOK):
            tok = int(want[i, j])
            assert rec[2 + 2 * TOK + j] == tok
            if tok >= 0:
                b, k = divmod(tok, N)
                mine = [(t * B + b) * ncap + slot[t, b, k] for t in range(nt) if stored[t, b, k]]
                assert rec[2 + j] == len(mine) and rec[2 + TOK + j] == kcount[b, k]
            else:
                mine = []
                assert rec[2 + j] == 0 and rec[2 + TOK + j] == 0
            rows += mine
        assert rec[1] == len(rows)
        assert rec[HEAD:HEAD + len(rows)].astype(np.uint32).tolist() == rows


@pytest.mark.parametrize("name", ["tiny", "small", "medium", "temporal", "large"])
def test_records_match_the_slot_path(tdp, name):
    wl = wk.by_name(name)
    plan, out, N, ncap = _setup(tdp, wl)
    recs, res = _blends(tdp, plan, wl, out, N, ncap)
    for _, O1, O2 in res:
        assert _same(O1, O2), "tdp_cond_blend_records differs from tdp_cond_blend"
    if name in ("tiny", "small", "medium"):
        _check_records(plan, wl, out, N, ncap, recs)


def test_records_with_half_the_tokens_kept_by_every_tile(tdp):
    """The large workload with half its tokens at negative time (kept by all 128 tiles): blocks
    of up to 1024 rows, many ring stages each."""
    wl = wk.by_name("large").replace(neg_frac=0.5)
    plan, out, N, ncap = _setup(tdp, wl)
    recs, res = _blends(tdp, plan, wl, out, N, ncap)
    for _, O1, O2 in res:
        assert _same(O1, O2)


@pytest.mark.parametrize("ncap", [1, 7])
def test_records_with_rows_past_capacity(tdp, ncap):
    wl = wk.by_name("small").replace(B=2, n_cond=1003)
    plan, out, N, ncap = _setup(tdp, wl, ncap=ncap)
    recs, res = _blends(tdp, plan, wl, out, N, ncap)
    for _, O1, O2 in res:
        assert _same(O1, O2)
    _check_records(plan, wl, out, N, ncap, recs)


def test_records_serve_many_calls(tdp):
    """One set of records, three calls with different per-tile outputs (the denoising loop)."""
    wl = wk.by_name("temporal")
    plan, out, N, ncap = _setup(tdp, wl)
    recs, res = _blends(tdp, plan, wl, out, N, ncap, seeds=(1, 2, 3))
    for _, O1, O2 in res:
        assert _same(O1, O2)


def test_records_against_the_oracle(tdp):
    wl = wk.by_name("small")
    plan, out, N, ncap = _setup(tdp, wl)
    recs, res = _blends(tdp, plan, wl, out, N, ncap)
    Yc, _, O2 = res[0]
    ref = oracle.cond_blend(oracle.problem_of(wl), to_host(Yc), out["keep"], out["idx"], out["count"], ncap)
    assert_blend_close(to_host(O2), ref, wl)


def test_records_wide_and_odd_channels(tdp):
    """bf16 C=136 (17 channel vectors: two slabs) and fp32, with a token kept by every tile."""
    for wl in (wk.by_name("tiny").replace(F=4, H=24, W=40, C=136, dtype="bf16", num_tiles=(2, 4, 8),
                                          overlap=(1, 2, 2), n_cond=400),
               wk.by_name("tiny").replace(n_cond=77)):
        plan, out, N, ncap = _setup(tdp, wl)
        recs, res = _blends(tdp, plan, wl, out, N, ncap)
        for _, O1, O2 in res:
            assert _same(O1, O2)


def test_records_at_the_tile_limit(tdp):
    """256 tiles (the most the records take), half the tokens with negative time."""
    wl = wk.by_name("tiny").replace(F=2, H=48, W=52, C=512, dtype="bf16", num_tiles=(1, 16, 16),
                                    overlap=(0, 1, 1), n_cond=120, neg_frac=0.5)
    plan, out, N, ncap = _setup(tdp, wl)
    assert plan.n_tiles == 256
    recs, res = _blends(tdp, plan, wl, out, N, ncap)
    for _, O1, O2 in res:
        assert _same(O1, O2)



def test_foreign_records_stay_in_bounds(tdp):
    """A buffer that does not hold records (random integers, huge row counts and row numbers):
    the outputs are meaningless, but nothing outside Ycond is read and nothing outside out is
    written (guard bands around out keep their bytes)."""
    import torch
    wl = wk.by_name("small")
    plan, out, N, ncap = _setup(tdp, wl)
    g = torch.Generator(device="cuda").manual_seed(5)
    n = tdp.tdp_cond_records_size(plan, N)
    recs = torch.randint(-2**31, 2**31 - 1, (n,), generator=g, device="cuda", dtype=torch.int64).to(torch.int32)
    Yc = to_dev(_storage(wl, (plan.n_tiles, wl.B, ncap, wl.C), 3))
    pad = 4096
    big = fill_sentinel(torch.empty(wl.B * N * wl.C + 2 * pad, dtype=torch.bfloat16, device="cuda"))
    ref = big.clone()
    tdp.tdp_cond_blend_records(plan, N, recs, Yc, ncap, big[pad:pad + wl.B * N * wl.C])
    torch.cuda.synchronize()
    assert _same(big[:pad], ref[:pad]) and _same(big[-pad:], ref[-pad:])
    # the same buffer with plausible block numbers: every record's number in [0, G)
    G = wl.B * ((N + TOK - 1) // TOK)
    stride = (HEAD + TOK * plan.n_tiles + 3) // 4 * 4
    r = recs[:G * stride].view(G, stride)
    r[:, 0] = torch.arange(G, device="cuda", dtype=torch.int32)
    tdp.tdp_cond_blend_records(plan, N, recs, Yc, ncap, big[pad:pad + wl.B * N * wl.C])
    torch.cuda.synchronize()
    assert _same(big[:pad], ref[:pad]) and _same(big[-pad:], ref[-pad:])
