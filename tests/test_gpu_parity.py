"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Split tiles, tile positions, position bounds, keep masks, compaction and
counts are compared bit for bit; the blend within the stated tolerance of the
fp64 oracle.  Source: "Tiled Data Parallelism (TDP)" (LTX-2 docs, multigpu).
"""
import numpy as np
import pytest

import oracle
import workloads as wk
from gpu_path import (as_f64, assert_blend_close, assert_filter_equal, fill_sentinel, run_blend,
                      run_split_filter, to_dev, to_host)

pytestmark = pytest.mark.gpu

FULL_ORACLE = ["tiny", "small", "medium", "temporal"]


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


def _plan(tdp, wl):
    return tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)


def _yout(wl, Y, seed):
    """Stand-in transformer output: tile + N(0, sigma), in the storage type."""
    noise = wk.make_noise(Y.shape, wl.sigma, np.random.default_rng(seed))
    if wl.dtype == "f32":
        return (Y + noise).astype(np.float32)
    return wk.f32_to_bf16_bits(wk.bf16_bits_to_f32(Y) + noise)


def _check_path(tdp, wl, X, P, K, normalize=True, stream=None):
    """Both forms of the pre-model stage (three calls, and tdp_split_filter) against the
    oracle, bit for bit; then the blend."""
    plan = _plan(tdp, wl)
    p = oracle.problem_of(wl)
    Yref, Qref = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Qref)
    Qn = oracle.normalize(p, Qref, mn) if normalize else Qref
    ref = dict(zip(("keep", "idx", "count", "kcount", "Kout", "slot"),
                   oracle.filter_cond(p, K, mn, mx, normalize, with_slot=True)))
    for fused in (False, True):
        out = run_split_filter(tdp, plan, wl, X, P, K, normalize=normalize, stream=stream, fused=fused)
        assert np.array_equal(out["Y"].reshape(Yref.shape), Yref), f"tile split differs (fused={fused})"
        assert np.array_equal(out["mn"], mn) and np.array_equal(out["mx"], mx), f"bounds differ (fused={fused})"
        assert np.array_equal(out["Q"], Qn), f"tile positions differ (fused={fused})"
        assert_filter_equal(out, ref, plan.n_tiles, wl.B)
    # blend of noisy tile outputs
    Yout = _yout(wl, Yref, wl.seed + 99)
    Z = run_blend(tdp, plan, wl, Yout, stream=stream)
    assert_blend_close(to_host(Z), oracle.blend(p, Yout), wl)
    # reconstruction: tile outputs equal to their tiles give back the latent
    Zr = to_host(run_blend(tdp, plan, wl, out["Yd"], stream=stream))
    if wl.dtype == "bf16":
        assert np.array_equal(Zr, X), "bf16 reconstruction is not bit-exact"
    else:
        assert np.allclose(Zr, X, rtol=1e-6, atol=1e-7)
    return plan


@pytest.mark.parametrize("name", FULL_ORACLE)
def test_parity_workload(tdp, name):
    wl = wk.by_name(name)
    X, P, K = wk.make_inputs(wl)
    _check_path(tdp, wl, X, P, K)


@pytest.mark.parametrize("name", ["tiny", "temporal"])
def test_parity_without_normalisation(tdp, name):
    wl = wk.by_name(name)
    X, P, K = wk.make_inputs(wl)
    _check_path(tdp, wl, X, P, K, normalize=False)


def test_parity_on_side_stream(tdp):
    import torch
    wl = wk.by_name("medium")
    X, P, K = wk.make_inputs(wl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _check_path(tdp, wl, X, P, K, stream=s)


def test_parity_edge_tokens(tdp):
    """Conditioning intervals that end on, or start just below, every tile edge; plus
    empty and inverted intervals."""
    wl = wk.by_name("temporal").replace(F=12, H=30, W=27, C=16, n_cond=3000)
    p = oracle.problem_of(wl)
    box, _ = oracle.plan(p)
    edges = [sorted(set(box[:, d, :].ravel().tolist())) for d in range(3)]
    rng = np.random.default_rng(5)
    X, P, _ = wk.make_inputs(wl)
    K = wk.make_cond_positions(wl, rng, edges=edges, edge_frac=0.5)
    K[:, 1, :40, 1] = K[:, 1, :40, 0]          # empty intervals
    K[:, 2, 40:80, 1] = K[:, 2, 40:80, 0] - 3  # inverted intervals
    _check_path(tdp, wl, X, P, K)


def test_parity_wrapping_positions(tdp):
    """Position values near the int32 limits: normalisation wraps the same way on both sides."""
    wl = wk.by_name("tiny").replace(F=4, H=10, W=12, n_cond=64)
    rng = np.random.default_rng(8)
    X, _, K = wk.make_inputs(wl)
    P = np.empty((wl.B, 3, wl.tokens, 2), np.int32)
    P[..., 0] = rng.integers(-2**31, 2**31 - 1, size=P.shape[:-1], dtype=np.int64).astype(np.int32)
    P[..., 1] = rng.integers(-2**31, 2**31 - 1, size=P.shape[:-1], dtype=np.int64).astype(np.int32)
    K[..., 0] = rng.integers(-2**31, 2**31 - 1, size=K.shape[:-1], dtype=np.int64).astype(np.int32)
    _check_path(tdp, wl, X, P, K)


@pytest.mark.parametrize("shape", [
    dict(num_tiles=(1, 1, 1), overlap=(0, 0, 0)),              # single tile: identity
    dict(num_tiles=(2, 3, 4), overlap=(0, 0, 0)),              # zero overlap: permutation
    dict(num_tiles=(2, 2, 2), overlap=(1, 1, 1)),              # odd overlap of one cell
    dict(num_tiles=(3, 2, 3), overlap=(3, 5, 3)),              # odd overlaps, uneven cores
    dict(H=32, W=40, num_tiles=(1, 2, 2), overlap=(0, 16, 20)),  # overlap == core: overlaps touch
    dict(F=3, H=8, W=12, num_tiles=(3, 8, 12), overlap=(1, 1, 0)),  # a tile per cell: one-cell cores
    dict(F=4, H=10, W=9, num_tiles=(2, 5, 3), overlap=(2, 2, 3)),   # overlap == core in every dimension
])
def test_parity_geometries(tdp, shape):
    base = wk.by_name("temporal").replace(F=9, H=26, W=30, C=24, n_cond=500)
    wl = base.replace(**shape)
    X, P, K = wk.make_inputs(wl)
    _check_path(tdp, wl, X, P, K)


def test_parity_max_tiles_per_dim(tdp):
    wl = wk.by_name("tiny").replace(F=2, H=6, W=130, C=8, dtype="bf16",
                                    num_tiles=(1, 3, 64), overlap=(0, 2, 1), n_cond=200)
    X, P, K = wk.make_inputs(wl)
    _check_path(tdp, wl, X, P, K)


def test_parity_minimal_rows(tdp):
    """16-byte tokens (bf16 C=8, fp32 C=4) and a one-cell-wide grid."""
    for wl in (wk.by_name("tiny").replace(C=8, dtype="bf16"),
               wk.by_name("tiny").replace(C=4),
               wk.by_name("tiny").replace(F=1, H=1, W=1, num_tiles=(1, 1, 1), overlap=(0, 0, 0))):
        X, P, K = wk.make_inputs(wl)
        _check_path(tdp, wl, X, P, K)


@pytest.mark.parametrize("fused", [False, True])
def test_no_cond_tokens(tdp, fused):
    wl = wk.by_name("small")
    X, P, _ = wk.make_inputs(wl)
    K = np.zeros((wl.B, 3, 0, 2), np.int32)
    plan = _plan(tdp, wl)
    out = run_split_filter(tdp, plan, wl, X, P, K, fused=fused)
    assert (out["count"] == 0).all()
    Yref, _ = oracle.split(oracle.problem_of(wl), X, P)
    assert np.array_equal(out["Y"].reshape(Yref.shape), Yref)


def test_split_without_positions(tdp):
    wl = wk.by_name("medium")
    X, P, K = wk.make_inputs(wl)
    plan = _plan(tdp, wl)
    out = run_split_filter(tdp, plan, wl, X, P, K, positions=False)
    Yref, _ = oracle.split(oracle.problem_of(wl), X, P)
    assert np.array_equal(out["Y"].reshape(Yref.shape), Yref)


def test_zero_batch(tdp):
    import torch
    wl = wk.by_name("tiny").replace(B=0)
    plan = _plan(tdp, wl)
    Y, Q, mn, mx = tdp.alloc_split_outputs(plan, "cuda")
    X = torch.empty((0, wl.F, wl.H, wl.W, wl.C), device="cuda")
    P = torch.empty((0, 3, wl.tokens, 2), dtype=torch.int32, device="cuda")
    tdp.tdp_pos_bounds(plan, P, mn, mx)
    tdp.tdp_split(plan, X, P, mn, 1, Y, Q)
    K = torch.empty((0, 3, 4, 2), dtype=torch.int32, device="cuda")
    keep, idx, count, kcount, Kout = tdp.alloc_filter_outputs(plan, 4, "cuda")
    tdp.tdp_split_filter(plan, X, P, K, 4, 1, Y, Q, mn, mx, keep, idx, count, kcount, Kout)
    Z = torch.empty_like(X)
    tdp.tdp_blend(plan, Y, Z)
    torch.cuda.synchronize()


def test_large_workload_in_bench_configuration(tdp):
    """The large workload at full size, as the benchmark launches it (tdp_split_filter, then
    tdp_blend), and through the three separate calls (tdp_pos_bounds, tdp_split,
    tdp_norm_filter): split and filter compared in full and bit for bit, the blend of noisy
    tile outputs element by element against the fp64 oracle over the whole latent, and the
    reconstruction property over every element."""
    import torch
    wl = wk.by_name("large")
    X, P, K = wk.make_inputs(wl)
    plan = _plan(tdp, wl)
    p = oracle.problem_of(wl)
    Yref, Qref = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Qref)
    Qn = oracle.normalize(p, Qref, mn)
    del Qref
    ref = dict(zip(("keep", "idx", "count", "kcount", "Kout", "slot"),
                   oracle.filter_cond(p, K, mn, mx, True, with_slot=True)))
    for fused in (False, True):
        out = run_split_filter(tdp, plan, wl, X, P, K, fused=fused)
        assert np.array_equal(out["Y"].reshape(Yref.shape), Yref), f"tile split differs (fused={fused})"
        assert np.array_equal(out["mn"], mn) and np.array_equal(out["mx"], mx), f"bounds differ (fused={fused})"
        assert np.array_equal(out["Q"], Qn), f"tile positions differ (fused={fused})"
        assert_filter_equal(out, ref, plan.n_tiles, wl.B)
        if not fused:
            del out
    del Yref, Qn
    # reconstruction over the whole latent
    Zr = run_blend(tdp, plan, wl, out["Yd"])
    assert torch.equal(Zr.view(torch.int16), to_dev(X).view(torch.int16))
    del Zr
    # noisy outputs, every element against the fp64 oracle (compared frame by frame)
    Yout = out["Yd"] + 0.05 * torch.randn(out["Yd"].shape, generator=torch.Generator("cuda").manual_seed(3),
                                          device="cuda", dtype=torch.float32).to(torch.bfloat16)
    Z = to_host(run_blend(tdp, plan, wl, Yout))
    Zref = oracle.blend(p, to_host(Yout))
    for f in range(wl.F):
        assert_blend_close(Z[:, f], Zref[:, f], wl)


def test_parity_wide_rows(tdp):
    """W above the blend's per-pass cell table (1024 cells): the table is rebuilt per pass."""
    wl = wk.by_name("tiny").replace(F=2, H=3, W=1100, C=16, dtype="bf16", num_tiles=(1, 1, 5),
                                    overlap=(0, 0, 8), n_cond=300)
    X, P, K = wk.make_inputs(wl)
    _check_path(tdp, wl, X, P, K)


def test_parity_many_cond_tokens(tdp):
    """More conditioning tokens than one compaction pass (16384) holds."""
    wl = wk.by_name("small").replace(B=2, n_cond=40000)
    X, P, K = wk.make_inputs(wl)
    _check_path(tdp, wl, X, P, K)


def test_parity_many_tiles(tdp):
    """2048 tiles: the keep counts stage tile bounds in shared memory in two rounds."""
    wl = wk.by_name("tiny").replace(F=4, H=64, W=64, C=8, dtype="bf16", num_tiles=(2, 32, 32),
                                    overlap=(1, 2, 1), n_cond=300)
    X, P, K = wk.make_inputs(wl)
    _check_path(tdp, wl, X, P, K)


def test_parity_wide_channels(tdp):
    """4 KB tokens (bf16 C=2048): 256 vectors per token."""
    wl = wk.by_name("tiny").replace(F=2, H=6, W=10, C=2048, dtype="bf16", num_tiles=(1, 2, 2),
                                    overlap=(0, 2, 2), n_cond=100)
    X, P, K = wk.make_inputs(wl)
    _check_path(tdp, wl, X, P, K)


def test_filter_keep_buffer_at_odd_address(tdp):
    """A keep buffer that starts one byte past a 16-byte boundary, with N a multiple of 16:
    the compaction reads keep bytes one at a time (its 16-byte loads need an aligned
    buffer, checked on the host), and every output still matches the oracle."""
    import torch
    wl = wk.by_name("small")
    X, P, K = wk.make_inputs(wl)
    plan = _plan(tdp, wl)
    p = oracle.problem_of(wl)
    N = K.shape[2]
    assert N % 16 == 0
    _, Qref = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Qref)
    ref = dict(zip(("keep", "idx", "count", "kcount", "Kout", "slot"),
                   oracle.filter_cond(p, K, mn, mx, True, with_slot=True)))
    nt, B = plan.n_tiles, wl.B
    raw = torch.full((nt * B * N + 16,), 0xAB, dtype=torch.uint8, device="cuda")
    keep = raw[1:1 + nt * B * N]
    assert keep.data_ptr() % 16 == 1
    _, idx, count, kcount, Kout, slot = tdp.alloc_filter_outputs(plan, N, "cuda", slot=True)
    tdp.tdp_norm_filter(plan, to_dev(K), N, to_dev(mn), to_dev(mx), 1, keep, idx, count, kcount, Kout, slot)
    torch.cuda.synchronize()
    out = dict(keep=to_host(keep).reshape(nt, B, N), idx=to_host(idx), count=to_host(count),
               kcount=to_host(kcount), Kout=to_host(Kout), slot=to_host(slot))
    assert_filter_equal(out, ref, nt, B)
    assert to_host(raw)[0] == 0xAB and (to_host(raw)[1 + nt * B * N:] == 0xAB).all()


@pytest.mark.parametrize("name", FULL_ORACLE + ["large"])
@pytest.mark.parametrize("normalize", [True, False])
def test_split_tma_parity(tdp, name, normalize):
    """tdp_split_tma (bulk-tensor loads of tile-row segments, bulk stores to every tile
    holding them, positions beside the copy) gives tdp_split's outputs bit for bit."""
    import torch
    wl = wk.by_name(name)
    X, P, K = wk.make_inputs(wl)
    plan = _plan(tdp, wl)
    p = oracle.problem_of(wl)
    Yref, Qref = oracle.split(p, X, P)
    mn, _ = oracle.bounds(p, Qref)
    Qexp = oracle.normalize(p, Qref, mn) if normalize else Qref
    Y, Q, _, _ = tdp.alloc_split_outputs(plan, "cuda")
    for t in (Y, Q):
        fill_sentinel(t)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):                     # twice: the second call runs over the first's outputs
        tdp.tdp_split_tma(plan, to_dev(X), to_dev(P), to_dev(mn), int(normalize), Y, Q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(to_host(Y).reshape(Yref.shape), Yref)
    assert np.array_equal(to_host(Q), Qexp)


def test_split_tma_without_positions_and_refusals(tdp):
    """Latent only (P = Q = NULL); and shapes past the tensor-map box limits are refused on
    the host with TDP_ERR_TOO_LARGE before any launch."""
    import torch
    wl = wk.by_name("medium")
    X, P, _ = wk.make_inputs(wl)
    plan = _plan(tdp, wl)
    Y, _, _, _ = tdp.alloc_split_outputs(plan, "cuda", positions=False)
    fill_sentinel(Y)
    tdp.tdp_split_tma(plan, to_dev(X), None, None, 1, Y, None)
    torch.cuda.synchronize()
    Yref, _ = oracle.split(oracle.problem_of(wl), X, P)
    assert np.array_equal(to_host(Y).reshape(Yref.shape), Yref)
    wide = wk.by_name("tiny").replace(F=2, H=3, W=40, C=512, dtype="bf16", num_tiles=(1, 1, 2), overlap=(0, 0, 2))
    pw = _plan(tdp, wide)
    Xw = torch.zeros((1, 2, 3, 40, 512), dtype=torch.bfloat16, device="cuda")
    Yw, _, _, _ = tdp.alloc_split_outputs(pw, "cuda", positions=False)
    with pytest.raises(tdp.TdpError, match="TDP_ERR_TOO_LARGE"):
        tdp.tdp_split_tma(pw, Xw, None, None, 1, Yw, None)


def test_split_tma_at_the_w_tile_limit(tdp):
    """64 W-tiles (the most a dimension takes) of one or two cells and f32 storage: the
    position warps' row tables are at their largest, the boxes at their smallest."""
    import torch
    wl = wk.by_name("tiny").replace(B=2, F=3, H=5, W=128, C=16, num_tiles=(1, 2, 64), overlap=(0, 1, 1), n_cond=8)
    X, P, _ = wk.make_inputs(wl)
    plan = _plan(tdp, wl)
    p = oracle.problem_of(wl)
    Yref, Qref = oracle.split(p, X, P)
    mn, _ = oracle.bounds(p, Qref)
    Y, Q, _, _ = tdp.alloc_split_outputs(plan, "cuda")
    for t in (Y, Q):
        fill_sentinel(t)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tdp.tdp_split_tma(plan, to_dev(X), to_dev(P), to_dev(mn), 1, Y, Q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(to_host(Y).reshape(Yref.shape), Yref)
    assert np.array_equal(to_host(Q), oracle.normalize(p, Qref, mn))
