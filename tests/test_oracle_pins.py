"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one oracle function against something fixed independently:
the stated tile size of the tiny workload, closed forms, exact-integer
invariants the method promises ("masks sum to 1 globally", "interval widths
are preserved", "negative-time tokens are kept by every tile"), numpy slicing
as an independent box extractor, and brute-force enumeration with exact
rationals on tiny grids.  Source: "Tiled Data Parallelism (TDP)" (LTX-2 docs,
multigpu), sections "What it is", "Position normalization", "Shared negative
(reference) positions" and "API / Tiling config".
"""
import itertools
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wk

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CPU_WORKLOADS = [w for w in wk.WORKLOADS if w.name in ("tiny", "small", "medium", "temporal")]


def _valid_1d(L, n, o):
    # balanced cores are floor(L/n) or ceil(L/n) long, so the shortest is floor(L/n)
    return L >= 1 and 1 <= n <= L and o >= 0 and (n == 1 or L // n >= o)


def _latent_f64(wl, X):
    return X.astype(np.float64) if wl.dtype == "f32" else wk.bf16_bits_to_f32(X).astype(np.float64)


# --------------------------------------------------------------------------- geometry
def test_tiny_tile_size_golden():
    fx = {}
    with open(os.path.join(GOLDEN, "tiny_tile_size.txt")) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                fx[k] = tuple(int(x) for x in v)
    p = oracle.problem(1, *fx["dims"], 16, 4, fx["num_tiles"], fx["overlap"])
    box, off = oracle.plan(p)
    sizes = box[:, :, 1] - box[:, :, 0]
    assert box.shape[0] == 4
    assert all(tuple(s) == fx["tile_size"] for s in sizes)
    assert off[-1] == 4 * 3 * 5 * 7


@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_boxes_closed_form(wl):
    for d in range(3):
        L, n, o = wl.dims[d], wl.num_tiles[d], wl.overlap[d]
        lo, hi = oracle.tile_boxes_1d(L, n, o)
        assert lo[0] == 0 and hi[n - 1] == L
        cover = np.zeros(L, int)
        for i in range(n):
            assert 0 <= lo[i] < hi[i] <= L
            cover[lo[i]:hi[i]] += 1
        if n > 1:
            # neighbours overlap by exactly o, and no cell lies in more than two tiles
            assert all(hi[i] - lo[i + 1] == o for i in range(n - 1))
        assert cover.min() >= 1 and cover.max() <= (2 if n > 1 and o > 0 else 1)
        assert (hi - lo).sum() == L + (n - 1) * (o if n > 1 else 0)


def test_boxes_validity_rule_sweep():
    for L in range(1, 26):
        for n in range(1, 9):
            for o in range(0, 7):
                ok = _valid_1d(L, n, o)
                if ok:
                    lo, hi = oracle.tile_boxes_1d(L, n, o)
                    # cores are balanced: lengths differ by at most one
                    cores = np.diff([(i * L) // n for i in range(n + 1)])
                    assert cores.max() - cores.min() <= 1
                else:
                    with pytest.raises(ValueError):
                        oracle.tile_boxes_1d(L, n, o)


@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_plan_offsets_are_prefix_sums(wl):
    p = oracle.problem_of(wl)
    box, off = oracle.plan(p)
    nF, nH, nW = wl.num_tiles
    assert box.shape[0] == nF * nH * nW
    sizes = np.prod(box[:, :, 1] - box[:, :, 0], axis=1)
    assert off[0] == 0 and np.array_equal(np.diff(off), sizes)
    # tile order is (iF*nH + iH)*nW + iW
    for t in range(box.shape[0]):
        iF, iH, iW = t // (nH * nW), (t // nW) % nH, t % nW
        for d, i in enumerate((iF, iH, iW)):
            lo, hi = oracle.tile_boxes_1d(wl.dims[d], wl.num_tiles[d], wl.overlap[d])
            assert tuple(box[t, d]) == (lo[i], hi[i])


# --------------------------------------------------------------------------- ramps / masks
def _sweep_geometries():
    for L in (1, 2, 5, 8, 12, 17, 32, 64):
        for n in (1, 2, 3, 4, 8):
            for o in (0, 1, 2, 3, 4, 8):
                if _valid_1d(L, n, o):
                    yield L, n, o


def test_ramps_partition_of_unity_exact():
    """'masks sum to 1 globally': per dimension the integer numerators sum to the denominator."""
    geos = list(_sweep_geometries()) + [(wl.dims[d], wl.num_tiles[d], wl.overlap[d])
                                        for wl in wk.WORKLOADS for d in range(3)]
    for L, n, o in geos:
        for x in range(L):
            nums = [oracle.ramp_num(L, n, o, i, x) for i in range(n)]
            den = nums[0][1]
            assert all(d == den for _, d in nums)
            assert sum(v for v, _ in nums) == den, (L, n, o, x)


def test_ramps_are_trapezoids():
    """Linear rise over the left overlap, flat top of 1, linear fall over the right overlap."""
    for L, n, o in _sweep_geometries():
        lo, hi = oracle.tile_boxes_1d(L, n, o)
        for i in range(n):
            vals = [oracle.ramp_num(L, n, o, i, x) for x in range(L)]
            num = np.array([v for v, _ in vals])
            den = vals[0][1]
            assert (num[:lo[i]] == 0).all() and (num[hi[i]:] == 0).all()
            inside = num[lo[i]:hi[i]]
            assert (inside > 0).all() and (inside <= den).all()
            rise = o if (i > 0 and n > 1) else 0
            fall = o if (i < n - 1 and n > 1) else 0
            if rise:
                assert np.array_equal(inside[:rise], np.arange(1, rise + 1))
            if fall:
                assert np.array_equal(inside[len(inside) - fall:], np.arange(fall, 0, -1))
            assert (inside[rise:len(inside) - fall] == den).all()


def test_ramp_mirror_symmetry():
    for L, n, o in _sweep_geometries():
        lo, hi = oracle.tile_boxes_1d(L, n, o)
        for i in range(n - 1):
            for k in range(o):
                a, _ = oracle.ramp_num(L, n, o, i, lo[i + 1] + k)
                b, _ = oracle.ramp_num(L, n, o, i + 1, hi[i] - 1 - k)
                assert a == b


def _exact_mask(wl, t, cell):
    nF, nH, nW = wl.num_tiles
    ii = (t // (nH * nW), (t // nW) % nH, t % nW)
    m = Fraction(1)
    for d in range(3):
        num, den = oracle.ramp_num(wl.dims[d], wl.num_tiles[d], wl.overlap[d], ii[d], cell[d])
        m *= Fraction(num, den)
    return m


def test_masks_sum_to_one_3d_bruteforce():
    small = [wk.by_name("tiny"),
             wk.by_name("tiny").replace(F=6, num_tiles=(2, 3, 2), overlap=(1, 1, 3)),
             wk.by_name("tiny").replace(F=5, H=7, W=9, num_tiles=(2, 2, 3), overlap=(2, 3, 2))]
    for wl in small:
        p = oracle.problem_of(wl)
        nt = int(np.prod(wl.num_tiles))
        for cell in itertools.product(range(wl.F), range(wl.H), range(wl.W)):
            exact = sum(_exact_mask(wl, t, cell) for t in range(nt))
            assert exact == 1
            approx = sum(oracle.mask(p, t, *cell) for t in range(nt))
            assert abs(approx - 1.0) < 1e-15
            for t in range(nt):
                assert oracle.mask(p, t, *cell) == float(_exact_mask(wl, t, cell)) or \
                    abs(oracle.mask(p, t, *cell) - float(_exact_mask(wl, t, cell))) < 1e-16


# --------------------------------------------------------------------------- split
@pytest.mark.parametrize("wl", CPU_WORKLOADS, ids=lambda w: w.name)
def test_split_matches_numpy_box_slicing(wl):
    X, P, K = wk.make_inputs(wl)
    p = oracle.problem_of(wl)
    box, off = oracle.plan(p)
    Y, Q = oracle.split(p, X, P)
    B, C = wl.B, wl.C
    P6 = P.reshape(B, 3, wl.F, wl.H, wl.W, 2)
    for t in range(box.shape[0]):
        (f0, f1), (h0, h1), (w0, w1) = box[t]
        Tt = int(off[t + 1] - off[t])
        yt = Y[B * off[t]:B * off[t + 1]].reshape(B, Tt, C)
        qt = Q[B * off[t] * 6:B * off[t + 1] * 6].reshape(B, 3, Tt, 2)
        ref_y = X[:, f0:f1, h0:h1, w0:w1, :].reshape(B, Tt, C)
        ref_q = P6[:, :, f0:f1, h0:h1, w0:w1, :].reshape(B, 3, Tt, 2)
        assert np.array_equal(yt.view(np.uint8), ref_y.view(np.uint8))
        assert np.array_equal(qt, ref_q)


def test_split_single_tile_is_identity():
    wl = wk.by_name("medium").replace(num_tiles=(1, 1, 1), overlap=(0, 0, 0))
    X, P, _ = wk.make_inputs(wl)
    Y, Q = oracle.split(oracle.problem_of(wl), X, P)
    assert np.array_equal(Y.reshape(X.shape), X)
    assert np.array_equal(Q.reshape(P.shape), P)


def test_split_zero_overlap_is_permutation():
    wl = wk.by_name("temporal").replace(F=8, H=20, W=24, C=16, overlap=(0, 0, 0))
    X, P, _ = wk.make_inputs(wl)
    # tag every token with its own flat index so a permutation is visible
    tag = np.arange(wl.B * wl.tokens, dtype=np.uint16).reshape(wl.B, wl.F, wl.H, wl.W, 1)
    Xt = np.broadcast_to(tag, X.shape).copy()
    Y, _ = oracle.split(oracle.problem_of(wl), Xt, P)
    assert Y.shape[0] == wl.B * wl.tokens
    assert np.array_equal(np.sort(Y[:, 0]), np.arange(wl.B * wl.tokens, dtype=np.uint16))


# --------------------------------------------------------------------------- bounds / normalisation
@pytest.mark.parametrize("wl", CPU_WORKLOADS, ids=lambda w: w.name)
def test_bounds_grid_positions_closed_form(wl):
    """With width-1 grid positions the tile's position extent is its box."""
    X, P, K = wk.make_inputs(wl)
    p = oracle.problem_of(wl)
    box, off = oracle.plan(p)
    _, Q = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Q)
    for b in range(wl.B):
        assert np.array_equal(mn[:, b, :], box[:, :, 0])
        assert np.array_equal(mx[:, b, :], box[:, :, 1])


def _tile_q(wl, Q, off, t):
    B = wl.B
    Tt = int(off[t + 1] - off[t])
    return Q[B * off[t] * 6:B * off[t + 1] * 6].reshape(B, 3, Tt, 2)


@pytest.mark.parametrize("wl", CPU_WORKLOADS, ids=lambda w: w.name)
def test_normalisation_grid_closed_form(wl):
    """Normalised grid positions of a tile are its local coordinates (f-lo_F, h-lo_H, w-lo_W)."""
    X, P, K = wk.make_inputs(wl)
    p = oracle.problem_of(wl)
    box, off = oracle.plan(p)
    _, Q = oracle.split(p, X, P)
    mn, _ = oracle.bounds(p, Q)
    Qn = oracle.normalize(p, Q, mn)
    for t in range(box.shape[0]):
        sz = box[t, :, 1] - box[t, :, 0]
        loc = np.stack([g.ravel() for g in np.meshgrid(*[np.arange(s) for s in sz], indexing="ij")])
        q = _tile_q(wl, Qn, off, t)
        for b in range(wl.B):
            assert np.array_equal(q[b, :, :, 0], loc)
            assert np.array_equal(q[b, :, :, 1], loc + 1)


def test_normalisation_invariants_random_positions():
    """Generated tokens start at 0 per (tile, batch, dim); every width is kept; kept cond
    tokens move by the tile's own offset."""
    wl = wk.by_name("temporal").replace(F=10, H=27, W=30, C=16, n_cond=300)
    rng = np.random.default_rng(7)
    X, _, K = wk.make_inputs(wl)
    P = np.empty((wl.B, 3, wl.tokens, 2), np.int32)
    P[..., 0] = rng.integers(-50, 200, size=P.shape[:-1])
    P[..., 1] = P[..., 0] + rng.integers(0, 9, size=P.shape[:-1])
    p = oracle.problem_of(wl)
    box, off = oracle.plan(p)
    _, Q = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Q)
    Qn = oracle.normalize(p, Q, mn)
    for t in range(box.shape[0]):
        q0, q1 = _tile_q(wl, Q, off, t), _tile_q(wl, Qn, off, t)
        assert (q1[..., 0].min(axis=2) == 0).all()
        assert np.array_equal(q1[..., 1] - q1[..., 0], q0[..., 1] - q0[..., 0])
        assert np.array_equal(q0[..., 0].min(axis=2), mn[t])
        assert np.array_equal(q0[..., 1].max(axis=2), mx[t])
    keep, idx, count, kcount, Kout = oracle.filter_cond(p, K, mn, mx, True)
    for t in range(box.shape[0]):
        for b in range(wl.B):
            c = count[t, b]
            ref = K[b][:, idx[t, b, :c], :] - mn[t, b][:, None, None]
            assert np.array_equal(Kout[t, b][:, :c, :], ref)


# --------------------------------------------------------------------------- conditioning filter
def _filter_bruteforce(wl, K, box):
    """Keep rule by enumeration of the tile's grid cells (valid for width-1 grid positions):
    an interval overlaps the tile in a dimension iff some cell coordinate of the tile lies in it."""
    nt = box.shape[0]
    N = K.shape[2]
    keep = np.zeros((nt, wl.B, N), np.uint8)
    for t in range(nt):
        for b in range(wl.B):
            for k in range(N):
                hit = True
                for d in range(3):
                    s, e = K[b, d, k]
                    if not any(s <= x < e for x in range(box[t, d, 0], box[t, d, 1])):
                        hit = False
                keep[t, b, k] = hit or K[b, 0, k, 0] < 0
    return keep


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_filter_bruteforce_and_compaction(name):
    wl = wk.by_name(name)
    p = oracle.problem_of(wl)
    box, off = oracle.plan(p)
    rng = np.random.default_rng(wl.seed + 17)
    edges = [sorted(set(box[:, d, :].ravel().tolist())) for d in range(3)]
    K = wk.make_cond_positions(wl, rng, n_cond=min(wl.n_cond, 400), edges=edges, edge_frac=0.3)
    X, P, _ = wk.make_inputs(wl)
    _, Q = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Q)
    keep, idx, count, kcount, Kout = oracle.filter_cond(p, K, mn, mx, True)
    assert np.array_equal(keep, _filter_bruteforce(wl, K, box))
    N = K.shape[2]
    for t in range(box.shape[0]):
        for b in range(wl.B):
            kept = np.nonzero(keep[t, b])[0]
            assert count[t, b] == len(kept)
            assert np.array_equal(idx[t, b, :len(kept)], kept)
            assert (idx[t, b, len(kept):] == -1).all()
    assert np.array_equal(kcount, keep.sum(axis=0))
    neg = K[:, 0, :, 0] < 0
    assert (kcount[neg] == box.shape[0]).all()
    # a token that covers at least one latent cell is kept by at least one tile
    L = np.array(wl.dims)
    covers = np.all((K[..., 0] < L[None, :, None]) & (K[..., 1] > 0), axis=1)
    assert (kcount[covers] >= 1).all()
    assert N == K.shape[2]


def test_filter_hand_built_edges():
    """Tokens placed on the edges of the tiny workload's tile (0,0,0) box [0,3)x[0,5)x[0,7)."""
    wl = wk.by_name("tiny")
    p = oracle.problem_of(wl)
    box, _ = oracle.plan(p)
    full = [(0, wl.F), (0, wl.H), (0, wl.W)]
    cases = []  # (interval per dim, expected keep for tile 0)
    lo, hi = box[0, 1]
    cases.append(([full[0], (lo - 2, lo), full[2]], False))   # ends exactly at the tile's start
    cases.append(([full[0], (hi - 1, hi + 3), full[2]], True))  # starts on the tile's last cell
    cases.append(([full[0], (hi, hi + 3), full[2]], False))     # starts just past the tile
    cases.append(([(-3, -1), (hi + 1, hi + 2), (40, 41)], True))  # negative time, far away
    cases.append(([(0, 1), (lo, lo + 1), (box[0, 2, 1] - 1, box[0, 2, 1])], True))  # corner cell
    cases.append(([(1, 1), full[1], full[2]], False))           # empty interval in time
    K = np.zeros((1, 3, len(cases), 2), np.int32)
    for k, (iv, _) in enumerate(cases):
        for d in range(3):
            K[0, d, k] = iv[d]
    X, P, _ = wk.make_inputs(wl)
    _, Q = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Q)
    keep, *_ = oracle.filter_cond(p, K, mn, mx, True)
    assert [bool(v) for v in keep[0, 0]] == [e for _, e in cases]


def test_filter_no_tokens():
    wl = wk.by_name("tiny")
    p = oracle.problem_of(wl)
    X, P, _ = wk.make_inputs(wl)
    _, Q = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Q)
    keep, idx, count, kcount, Kout = oracle.filter_cond(p, np.zeros((1, 3, 0, 2), np.int32), mn, mx)
    assert keep.size == 0 and (count == 0).all()


# --------------------------------------------------------------------------- blend
@pytest.mark.parametrize("wl", CPU_WORKLOADS, ids=lambda w: w.name)
def test_blend_reconstructs_input(wl):
    """If every tile output equals its extracted tile, the blend gives back the latent."""
    X, P, _ = wk.make_inputs(wl)
    p = oracle.problem_of(wl)
    Y, _ = oracle.split(p, X, P)
    Z = oracle.blend(p, Y)
    ref = _latent_f64(wl, X)
    assert np.max(np.abs(Z - ref)) <= 1e-14 * max(1.0, np.max(np.abs(ref)))


def test_blend_zero_overlap_is_exact_inverse():
    wl = wk.by_name("temporal").replace(F=8, H=20, W=24, C=8, overlap=(0, 0, 0))
    X, P, _ = wk.make_inputs(wl)
    p = oracle.problem_of(wl)
    Y, _ = oracle.split(p, X, P)
    assert np.array_equal(oracle.blend(p, Y), _latent_f64(wl, X))


def test_blend_exact_rational_bruteforce():
    wl = wk.by_name("tiny").replace(F=4, C=3, num_tiles=(2, 2, 2), overlap=(1, 2, 2))
    p = oracle.problem_of(wl)
    box, off = oracle.plan(p)
    rng = np.random.default_rng(3)
    Yout = rng.integers(-64, 64, size=(wl.B * int(off[-1]), wl.C)).astype(np.float32) / 8
    Z = oracle.blend(p, Yout)
    for cell in itertools.product(range(wl.F), range(wl.H), range(wl.W)):
        acc = [Fraction(0)] * wl.C
        for t in range(box.shape[0]):
            if all(box[t, d, 0] <= cell[d] < box[t, d, 1] for d in range(3)):
                sz = box[t, :, 1] - box[t, :, 0]
                loc = [cell[d] - box[t, d, 0] for d in range(3)]
                j = (loc[0] * sz[1] + loc[1]) * sz[2] + loc[2]
                m = _exact_mask(wl, t, cell)
                row = Yout[off[t] + j]
                acc = [a + m * Fraction(float(v)) for a, v in zip(acc, row)]
        got = Z[0, cell[0], cell[1], cell[2]]
        assert np.allclose(got, [float(a) for a in acc], rtol=1e-15, atol=1e-15)


def test_blend_is_linear():
    wl = wk.by_name("tiny")
    p = oracle.problem_of(wl)
    _, off = oracle.plan(p)
    rng = np.random.default_rng(11)
    shape = (wl.B * int(off[-1]), wl.C)
    a = rng.integers(-100, 100, size=shape).astype(np.float32)
    b = rng.integers(-100, 100, size=shape).astype(np.float32)
    za, zb, zab = oracle.blend(p, a), oracle.blend(p, b), oracle.blend(p, a + b)
    assert np.max(np.abs(zab - (za + zb))) < 1e-11


def test_blend_cell_matches_blend():
    wl = wk.by_name("small")
    p = oracle.problem_of(wl)
    X, P, _ = wk.make_inputs(wl)
    Y, _ = oracle.split(p, X, P)
    noise = wk.make_noise(Y.shape, 0.05, np.random.default_rng(5))
    Yout = wk.f32_to_bf16_bits(wk.bf16_bits_to_f32(Y) + noise)
    Z = oracle.blend(p, Yout)
    rng = np.random.default_rng(6)
    for _ in range(40):
        f, h, w = (int(rng.integers(0, L)) for L in wl.dims)
        assert np.array_equal(oracle.blend_cell(p, Yout, 0, f, h, w), Z[0, f, h, w])


def test_oracle_is_independent_of_cuda_path():
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for fn in os.listdir(os.path.join(here, "oracle")):
        if fn.endswith((".py", ".c", ".h")):
            src = open(os.path.join(here, "oracle", fn)).read()
            assert "import blend_tdp_tile_gb300" not in src
            assert "from blend_tdp_tile_gb300" not in src
            assert "#include \"tdp.h\"" not in src and "libtdp" not in src


# --------------------------------------------------------------------------- conditioning outputs / audio
def _filtered(wl, n_cond=None, seed=21):
    p = oracle.problem_of(wl)
    X, P, _ = wk.make_inputs(wl)
    K = wk.make_cond_positions(wl, np.random.default_rng(seed), n_cond=n_cond)
    _, Q = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Q)
    keep, idx, count, kcount, Kout, slot = oracle.filter_cond(p, K, mn, mx, True, with_slot=True)
    return p, K, keep, idx, count, kcount, slot


def test_slot_is_inverse_of_compaction():
    wl = wk.by_name("small")
    p, K, keep, idx, count, kcount, slot = _filtered(wl, n_cond=300)
    for t in range(keep.shape[0]):
        for b in range(wl.B):
            c = count[t, b]
            assert np.array_equal(slot[t, b, idx[t, b, :c]], np.arange(c))
            assert (slot[t, b][keep[t, b] == 0] == -1).all()


@pytest.mark.parametrize("name", ["tiny", "small", "temporal"])
def test_cond_blend_identity_outputs_give_back_features(name):
    """If every tile returns each kept token's own feature, the average over the keeping
    tiles is that feature; a token no tile kept gets 0."""
    wl = wk.by_name(name).replace(n_cond=min(wk.by_name(name).n_cond, 600))
    p, K, keep, idx, count, kcount, slot = _filtered(wl)
    nt, N = keep.shape[0], keep.shape[2]
    feat = (np.random.default_rng(2).integers(-64, 64, size=(wl.B, N, wl.C)) / 16).astype(np.float32)
    Yc = np.zeros((nt, wl.B, N, wl.C), np.float32)
    for t in range(nt):
        for b in range(wl.B):
            c = count[t, b]
            Yc[t, b, :c] = feat[b, idx[t, b, :c]]
    if wl.dtype == "bf16":
        Yc = wk.f32_to_bf16_bits(Yc)       # features are exact in bf16 (multiples of 1/16, |x| <= 4)
    out = oracle.cond_blend(p, Yc, keep, idx, count, N)
    kept = kcount > 0
    assert np.allclose(out[kept], feat[kept], rtol=0, atol=1e-12)
    assert (out[~kept] == 0).all()


def test_cond_blend_constant_per_tile_outputs():
    """Tile t returning the constant t for every token: the result is the mean tile index
    over the keeping tiles, and (n_tiles-1)/2 for negative-time tokens."""
    wl = wk.by_name("temporal").replace(n_cond=500)
    p, K, keep, idx, count, kcount, slot = _filtered(wl)
    nt, N = keep.shape[0], keep.shape[2]
    Yc = np.broadcast_to(np.arange(nt, dtype=np.float32)[:, None, None, None], (nt, wl.B, N, wl.C)).copy()
    out = oracle.cond_blend(p, wk.f32_to_bf16_bits(Yc), keep, idx, count, N)
    tiles = np.arange(nt, dtype=np.float64)[:, None, None]
    with np.errstate(invalid="ignore", divide="ignore"):
        expect = (keep * tiles).sum(axis=0) / kcount
    kept = kcount > 0
    assert np.allclose(out[..., 0][kept], expect[kept], rtol=0, atol=1e-12)
    neg = K[:, 0, :, 0] < 0
    assert np.allclose(out[..., 0][neg], (nt - 1) / 2, atol=1e-12)


def test_cond_blend_single_keeper_is_exact_and_linear():
    wl = wk.by_name("small").replace(n_cond=400)
    p, K, keep, idx, count, kcount, slot = _filtered(wl)
    nt, N = keep.shape[0], keep.shape[2]
    rng = np.random.default_rng(4)
    a = rng.integers(-100, 100, size=(nt, wl.B, N, wl.C)).astype(np.float32)
    b = rng.integers(-100, 100, size=(nt, wl.B, N, wl.C)).astype(np.float32)
    wl32 = wl.replace(dtype="f32")
    p32 = oracle.problem_of(wl32)
    oa, ob, oab = (oracle.cond_blend(p32, x, keep, idx, count, N) for x in (a, b, a + b))
    assert np.max(np.abs(oab - (oa + ob))) < 1e-9
    one = kcount == 1
    for bb, k in zip(*np.nonzero(one)):
        t = int(np.nonzero(keep[:, bb, k])[0][0])
        assert np.array_equal(oa[bb, k], a[t, bb, slot[t, bb, k]].astype(np.float64))


def test_cond_blend_rows_past_capacity_keep_the_page_weight():
    """Hand-built case with one stored row per (tile, batch item) (ncap = 1), fixed by hand.
    Four tiles, four tokens; token 3 is kept by every tile but stored only by tile 1 (its
    only kept token there).  The page's weight is 1/(tiles that kept it) = 1/4, so its
    output is tile 1's row / 4, not tile 1's row alone; the other tokens have one keeper
    each and come back whole."""
    p = oracle.problem(1, 1, 8, 8, 4, 4, (1, 2, 2), (0, 2, 2))      # fp32, C = 4, 4 tiles
    N, ncap = 4, 1
    kept = {0: [0, 3], 1: [3], 2: [1, 3], 3: [2, 3]}                  # tile -> kept tokens
    keep = np.zeros((4, 1, N), np.uint8)
    idx = np.full((4, 1, N), -1, np.int32)
    count = np.zeros((4, 1), np.int32)
    for t, ks in kept.items():
        keep[t, 0, ks] = 1
        idx[t, 0, :len(ks)] = ks
        count[t, 0] = len(ks)
    base = np.array([1.0, 2.0, 3.0, 4.0], np.float32)
    Yc = np.stack([(t + 1) * base for t in range(4)]).reshape(4, 1, ncap, 4).astype(np.float32)
    out = oracle.cond_blend(p, Yc, keep, idx, count, ncap)
    expect = np.array([[1.0, 2.0, 3.0, 4.0],       # token 0: tile 0 only, row 0
                       [3.0, 6.0, 9.0, 12.0],      # token 1: tile 2 only, row 0
                       [4.0, 8.0, 12.0, 16.0],     # token 2: tile 3 only, row 0
                       [0.5, 1.0, 1.5, 2.0]])      # token 3: 4 keepers, one stored row (tile 1: 2*base) / 4
    assert np.array_equal(out[0], expect)


def test_tile_mean_pins():
    wl = wk.by_name("temporal")
    p = oracle.problem_of(wl.replace(dtype="f32"))
    nt, L = int(np.prod(wl.num_tiles)), 96
    const = np.broadcast_to(np.arange(nt, dtype=np.float32)[:, None, None], (nt, wl.B, L)).copy()
    assert np.allclose(oracle.tile_mean(p, const, L), (nt - 1) / 2, atol=1e-12)
    same = np.broadcast_to(np.random.default_rng(1).standard_normal((1, wl.B, L), dtype=np.float32),
                           (nt, wl.B, L)).copy()
    assert np.allclose(oracle.tile_mean(p, same, L), same[0].astype(np.float64), rtol=1e-14, atol=1e-15)
    one = oracle.problem_of(wl.replace(dtype="f32", num_tiles=(1, 1, 1), overlap=(0, 0, 0)))
    x = np.random.default_rng(3).standard_normal((1, wl.B, L), dtype=np.float32)
    assert np.array_equal(oracle.tile_mean(one, x, L), x[0].astype(np.float64))
