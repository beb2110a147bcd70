"""Maximum sizes: buffers past 2^31 elements and 4 GiB, where an index computed in
32 bits would wrap.

- Split and blend: a 2.18 G-element latent (4.4 GB bf16) in tiles whose buffer holds
  3.1 G elements (6.2 GB).
  - Position bounds and the conditioning filter are compared in full with the oracle.
  - Tile rows and tile positions are compared on sampled tokens, each against the
    latent cell the oracle's tile boxes put there. The samples include the first and
    last token of every tile.
  - The blend is compared on sampled cells, each computed alone by the oracle. Every
    element is also checked by the reconstruction property blend(split(X)) == X.
- Tile mean: inputs of 2.3 G elements, compared on sampled columns (the mean over
  tiles is columnwise, so the oracle runs on the gathered columns alone).
- Conditioning blend: rows of Ycond reserved so that the last tiles' kept rows sit
  past element 2^31.

Method: "Tiled Data Parallelism (TDP)" (LTX-2 docs, multigpu), "What it is",
"Position normalization", "Shared negative (reference) positions".
"""
import numpy as np
import pytest

import oracle
import workloads as wk
from gpu_path import assert_blend_close, assert_filter_equal, run_split_filter, to_dev, to_host

pytestmark = pytest.mark.gpu

TWO31 = 1 << 31


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


def _plan(tdp, wl):
    return tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)


def _rows(t, idx):
    """Rows `idx` of a 2-D device tensor, on the host (bf16 as uint16 bits)."""
    import torch
    return to_host(t.index_select(0, torch.as_tensor(np.asarray(idx, np.int64), device=t.device)))


def test_split_and_blend_past_32bit_offsets(tdp):
    import torch
    wl = wk.by_name("large").replace(F=16, H=512, W=1040, C=256, num_tiles=(2, 4, 4), overlap=(4, 16, 16),
                                     n_cond=4096)
    B, C = wl.B, wl.C
    T = wl.tokens
    assert B * T * C > TWO31
    plan = _plan(tdp, wl)
    p = oracle.problem_of(wl)
    box, off = oracle.plan(p)
    nt, tot = plan.n_tiles, plan.total_tile_tokens
    assert tot == int(off[-1]) and B * tot * C > TWO31
    rng = np.random.default_rng(wl.seed)
    P = wk.make_gen_positions(wl)
    K = wk.make_cond_positions(wl, rng)
    N = K.shape[2]
    gen = torch.Generator("cuda").manual_seed(wl.seed)
    X = torch.randn((B, wl.F, wl.H, wl.W, C), generator=gen, device="cuda", dtype=torch.bfloat16)
    Y, Q, mn, mx = tdp.alloc_split_outputs(plan, "cuda")
    Y.fill_(float("nan"))
    keep, idx, count, kcount, Kout, slot = tdp.alloc_filter_outputs(plan, N, "cuda", slot=True)
    tdp.tdp_split_filter(plan, X, to_dev(P), to_dev(K), N, 1, Y, Q, mn, mx, keep, idx, count, kcount, Kout, slot)
    torch.cuda.synchronize()

    # grid positions: each tile's bounds are its box (a closed form of the oracle's bounds)
    mn_ref = np.broadcast_to(box[:, None, :, 0], (nt, B, 3)).astype(np.int32)
    mx_ref = np.broadcast_to(box[:, None, :, 1], (nt, B, 3)).astype(np.int32)
    assert np.array_equal(to_host(mn), mn_ref) and np.array_equal(to_host(mx), mx_ref)
    ref = dict(zip(("keep", "idx", "count", "kcount", "Kout", "slot"),
                   oracle.filter_cond(p, K, mn_ref, mx_ref, True, with_slot=True)))
    out = {k: to_host(v) for k, v in dict(keep=keep, idx=idx, count=count, kcount=kcount, Kout=Kout,
                                          slot=slot).items()}
    assert_filter_equal(out, ref, nt, B)

    # sampled tile tokens: first and last of every tile, and random ones
    srng = np.random.default_rng(5)
    picks = []
    for t in range(nt):
        Tt = int(off[t + 1] - off[t])
        picks += [(t, 0), (t, Tt - 1)] + [(t, int(j)) for j in srng.integers(0, Tt, 12)]
    yrows, xrows, qexp, qidx = [], [], [], []
    for t, j in picks:
        sF, sH, sW = (int(box[t, d, 1] - box[t, d, 0]) for d in range(3))
        jf, jh, jw = j // (sH * sW), (j // sW) % sH, j % sW
        f, h, w = box[t, 0, 0] + jf, box[t, 1, 0] + jh, box[t, 2, 0] + jw
        Tt = int(off[t + 1] - off[t])
        yrows.append(B * int(off[t]) + j)                     # batch item 0
        xrows.append((int(f) * wl.H + int(h)) * wl.W + int(w))
        for d, v in enumerate((jf, jh, jw)):
            for s in range(2):
                qidx.append(((B * int(off[t])) * 3 + d * Tt + j) * 2 + s)
                qexp.append(v + s)
    assert max(yrows) * C > TWO31
    assert np.array_equal(_rows(Y, yrows), _rows(X.view(B * T, C), xrows)), "sampled tile rows differ"
    assert np.array_equal(to_host(Q[torch.as_tensor(qidx, device="cuda")]), np.asarray(qexp, np.int32))

    # reconstruction over every element
    Z = torch.empty_like(X)
    Z.fill_(float("nan"))
    tdp.tdp_blend(plan, Y, Z)
    torch.cuda.synchronize()
    assert torch.equal(Z.view(torch.int16), X.view(torch.int16)), "blend(split(X)) != X"

    # perturbed tile outputs, sampled cells against the oracle's per-cell blend
    Yout = Y
    Yout.add_(torch.randn(Y.shape, generator=gen, device="cuda", dtype=torch.bfloat16), alpha=0.05)
    Z.fill_(float("nan"))
    tdp.tdp_blend(plan, Yout, Z)
    torch.cuda.synchronize()
    del X
    cells = [(0, 0, 0), (wl.F - 1, wl.H - 1, wl.W - 1), (wl.F - 1, wl.H - 1, 0), (wl.F - 1, 0, wl.W - 1)]
    for d in range(3):
        for v in np.unique(box[:, d, :]):
            c = [int(srng.integers(0, L)) for L in wl.dims]
            c[d] = min(int(v), wl.dims[d] - 1)
            cells.append(tuple(c))
    cells += [tuple(int(srng.integers(0, L)) for L in wl.dims) for _ in range(200)]
    zrows = _rows(Z.view(B * T, C), [(f * wl.H + h) * wl.W + w for f, h, w in cells])
    del Z
    Yout_h = to_host(Yout)
    del Yout, Y
    for (f, h, w), z in zip(cells, zrows):
        assert_blend_close(z, oracle.blend_cell(p, Yout_h, 0, f, h, w), wl)


def test_tile_mean_past_32bit_offsets(tdp):
    import torch
    wl = wk.by_name("small").replace(num_tiles=(2, 4, 4), overlap=(2, 8, 8))
    plan = _plan(tdp, wl)
    nt = plan.n_tiles
    L = 72_000_000
    assert nt * wl.B * L > TWO31
    gen = torch.Generator("cuda").manual_seed(11)
    A = torch.randn((nt, wl.B, L), generator=gen, device="cuda", dtype=torch.bfloat16)
    out = torch.full((wl.B, L), float("nan"), device="cuda", dtype=torch.bfloat16)
    tdp.tdp_tile_mean(plan, L, A, out)
    torch.cuda.synchronize()
    srng = np.random.default_rng(12)
    cols = np.unique(np.concatenate([np.arange(8), np.arange(L - 8, L), srng.integers(0, L, 2000)]))
    ci = torch.as_tensor(cols, device="cuda")
    As = to_host(A.index_select(2, ci).contiguous())
    ref = oracle.tile_mean(oracle.problem_of(wl), As, len(cols))
    assert_blend_close(to_host(out.index_select(1, ci).contiguous()), ref, wl)


def test_cond_blend_past_32bit_offsets(tdp):
    import torch
    wl = wk.by_name("small").replace(num_tiles=(2, 4, 4), overlap=(2, 8, 8), n_cond=2048)
    X, P, K = wk.make_inputs(wl)
    plan = _plan(tdp, wl)
    nt, B, C, N = plan.n_tiles, wl.B, wl.C, K.shape[2]
    res = run_split_filter(tdp, plan, wl, X, P, K, fused=True)
    ncap = 600_000                      # rows reserved per (tile, batch): tile 31 starts past 2^31 elements
    assert (nt - 1) * B * ncap * C > TWO31
    gen = torch.Generator("cuda").manual_seed(13)
    Yc = torch.randn((nt, B, ncap, C), generator=gen, device="cuda", dtype=torch.bfloat16)
    out = torch.full((B, N, C), float("nan"), device="cuda", dtype=torch.bfloat16)
    tdp.tdp_cond_blend(plan, N, ncap, Yc, res["slotd"], out)
    torch.cuda.synchronize()
    used = max(1, int(res["count"].max()))
    Ys = to_host(Yc[:, :, :used].contiguous())           # rows at or past a tile's count are never read
    del Yc
    ref = oracle.cond_blend(oracle.problem_of(wl), Ys, res["keep"], res["idx"], res["count"], used)
    assert_blend_close(to_host(out), ref, wl)
