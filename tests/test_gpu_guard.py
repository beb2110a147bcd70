"""Out-of-range accesses, checked without a memory checker.

Every buffer an entry point takes lives inside a larger device allocation with a
guard band of GUARD bytes on each side:
- an output's bands hold a byte pattern that must be unchanged after the call
  (a write past either end of the output shows up there);
- an input's bands hold 0xFF bytes (NaN for f32/bf16, -1 for int32), so a kernel
  that read past an input and used what it found would change a result, and the
  element-by-element comparison with the CPU oracle would fail.

Each case runs every entry point: tdp_pos_bounds, tdp_split, tdp_split_tma,
tdp_norm_filter, tdp_split_filter, tdp_blend, tdp_cond_blend, tdp_cond_records and
tdp_cond_blend_records (where the tiles are 256 or fewer), tdp_blend_cond and
tdp_tile_mean, on ragged
geometries (tails in every dimension, several batch items, minimal and odd
channel counts).  Method: "Tiled Data Parallelism (TDP)" (LTX-2 docs, multigpu).
"""
import numpy as np
import pytest

import oracle
import workloads as wk
from gpu_path import assert_blend_close, assert_filter_equal, to_host

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes each side; a multiple of 256 keeps every view's alignment
OUT_FILL = 0xA5
IN_FILL = 0xFF


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


class Guarded:
    """A tensor of `shape`/`dtype` at byte offset GUARD inside a filled uint8 allocation."""

    def __init__(self, shape, dtype, fill):
        import torch
        self.fill = fill
        self.nbytes = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        self.raw = torch.full((2 * GUARD + self.nbytes,), fill, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def bands_intact(self) -> bool:
        lo = self.raw[:GUARD]
        hi = self.raw[GUARD + self.nbytes:]
        return bool((lo == self.fill).all()) and bool((hi == self.fill).all())


def _input(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        src = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        src = torch.from_numpy(a)
    g = Guarded(tuple(a.shape), src.dtype, IN_FILL)
    g.t.copy_(src)
    return g


def _output(shape, dtype):
    return Guarded(tuple(shape), dtype, OUT_FILL)


def _check_bands(bufs: dict, where: str):
    bad = [k for k, g in bufs.items() if not g.bands_intact()]
    assert not bad, f"{where}: guard bands changed around {bad}"


def _lat(wl):
    import torch
    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def _host(g):
    return to_host(g.t)


CASES = [
    ("tiny f32", wk.by_name("tiny")),
    ("tiny bf16 C=8", wk.by_name("tiny").replace(C=8, dtype="bf16")),
    ("f32 C=4, ragged", wk.by_name("tiny").replace(B=2, F=5, H=11, W=13, C=4, num_tiles=(2, 3, 2),
                                                     overlap=(1, 2, 3), n_cond=77)),
    ("bf16 C=24, two batch items", wk.by_name("temporal").replace(F=9, H=26, W=30, C=24, n_cond=500)),
    ("bf16 C=136, one-cell cores", wk.by_name("small").replace(B=2, F=3, H=8, W=12, C=136, num_tiles=(3, 8, 12),
                                                                 overlap=(1, 1, 0), n_cond=301)),
]


@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_guard_bands(tdp, name, wl):
    import torch
    i32, u8, lat = torch.int32, torch.uint8, _lat(wl)
    plan = tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)
    nt, B, C, tot = plan.n_tiles, wl.B, wl.C, plan.total_tile_tokens
    p = oracle.problem_of(wl)
    X, P, K = wk.make_inputs(wl)
    N = K.shape[2]
    Yref, Qref = oracle.split(p, X, P)
    mnr, mxr = oracle.bounds(p, Qref)
    Qn = oracle.normalize(p, Qref, mnr)
    ref = dict(zip(("keep", "idx", "count", "kcount", "Kout", "slot"),
                   oracle.filter_cond(p, K, mnr, mxr, True, with_slot=True)))
    Xg, Pg, Kg = _input(X), _input(P), _input(K)

    def split_outputs():
        return dict(Y=_output((B * tot, C), lat), Q=_output((B * tot * 6,), i32),
                    mn=_output((nt, B, 3), i32), mx=_output((nt, B, 3), i32),
                    keep=_output((nt, B, N), u8), idx=_output((nt, B, N), i32),
                    count=_output((nt, B), i32), kcount=_output((B, N), i32),
                    Kout=_output((nt, B, 3, N, 2), i32), slot=_output((nt, B, N), i32))

    def check_split(o, where):
        _check_bands(o, where)
        assert np.array_equal(_host(o["Y"]).reshape(Yref.shape), Yref), where
        assert np.array_equal(_host(o["Q"]), Qn), where
        assert np.array_equal(_host(o["mn"]), mnr) and np.array_equal(_host(o["mx"]), mxr), where
        assert_filter_equal({k: _host(o[k]) for k in ref}, ref, nt, B)

    # three calls
    o = split_outputs()
    tdp.tdp_pos_bounds(plan, Pg.t, o["mn"].t, o["mx"].t)
    tdp.tdp_split(plan, Xg.t, Pg.t, o["mn"].t, 1, o["Y"].t, o["Q"].t)
    tdp.tdp_norm_filter(plan, Kg.t, N, o["mn"].t, o["mx"].t, 1, o["keep"].t, o["idx"].t, o["count"].t,
                        o["kcount"].t, o["Kout"].t, o["slot"].t)
    torch.cuda.synchronize()
    check_split(o, "separate calls")

    # one call
    o = split_outputs()
    tdp.tdp_split_filter(plan, Xg.t, Pg.t, Kg.t, N, 1, o["Y"].t, o["Q"].t, o["mn"].t, o["mx"].t, o["keep"].t,
                         o["idx"].t, o["count"].t, o["kcount"].t, o["Kout"].t, o["slot"].t)
    torch.cuda.synchronize()
    check_split(o, "tdp_split_filter")

    # the latent moved by bulk-tensor loads and bulk stores (positions beside it)
    o = dict(Y=_output((B * tot, C), lat), Q=_output((B * tot * 6,), i32), err=_output((1,), i32))
    o["err"].t.zero_()
    mn_in = _input(mnr)
    tdp.tdp_split_tma(plan, Xg.t, Pg.t, mn_in.t, 1, o["Y"].t, o["Q"].t, o["err"].t)
    torch.cuda.synchronize()
    _check_bands(o, "tdp_split_tma")
    assert int(o["err"].t.item()) == 0, "tdp_split_tma: a bulk-tensor load timed out"
    assert np.array_equal(_host(o["Y"]).reshape(Yref.shape), Yref), "tdp_split_tma"
    assert np.array_equal(_host(o["Q"]), Qn), "tdp_split_tma"

    # blend of perturbed tile outputs
    noise = wk.make_noise(Yref.shape, wl.sigma, np.random.default_rng(wl.seed + 7))
    Yout = ((Yref + noise).astype(np.float32) if wl.dtype == "f32"
            else wk.f32_to_bf16_bits(wk.bf16_bits_to_f32(Yref) + noise))
    Yg = _input(Yout.reshape(B * tot, C))
    Zg = _output((B, wl.F, wl.H, wl.W, C), lat)
    tdp.tdp_blend(plan, Yg.t, Zg.t)
    torch.cuda.synchronize()
    _check_bands({"Z": Zg}, "tdp_blend")
    assert_blend_close(_host(Zg), oracle.blend(p, Yout), wl)

    # conditioning blend over the filter's slots
    ncap = max(1, int(ref["count"].max()))
    Yc = np.random.default_rng(wl.seed + 8).standard_normal((nt, B, ncap, C), dtype=np.float32)
    Yc = Yc if wl.dtype == "f32" else wk.f32_to_bf16_bits(Yc)
    Ycg, Sg = _input(Yc), _input(ref["slot"])
    Rg = _output((B, N, C), lat)
    tdp.tdp_cond_blend(plan, N, ncap, Ycg.t, Sg.t, Rg.t)
    torch.cuda.synchronize()
    _check_bands({"out": Rg}, "tdp_cond_blend")
    assert_blend_close(_host(Rg), oracle.cond_blend(p, Yc, ref["keep"], ref["idx"], ref["count"], ncap), wl)

    # the same outputs from per-block records (the records take at most 256 tiles)
    if nt <= 256:
        Rec = _output((tdp.tdp_cond_records_size(plan, N),), i32)
        tdp.tdp_cond_records(plan, N, ncap, Sg.t, Rec.t)
        Rg3 = _output((B, N, C), lat)
        tdp.tdp_cond_blend_records(plan, N, Rec.t, Ycg.t, ncap, Rg3.t)
        torch.cuda.synchronize()
        _check_bands({"recs": Rec, "out": Rg3}, "tdp_cond_records / tdp_cond_blend_records")
        assert np.array_equal(_host(Rg3), _host(Rg)), "tdp_cond_blend_records"

    # the post-model stage in one call: the same bytes as the two calls above
    Zg2, Rg2 = _output((B, wl.F, wl.H, wl.W, C), lat), _output((B, N, C), lat)
    tdp.tdp_blend_cond(plan, Yg.t, Zg2.t, N, ncap, Ycg.t, Sg.t, Rg2.t)
    torch.cuda.synchronize()
    _check_bands({"Z": Zg2, "out": Rg2}, "tdp_blend_cond")
    assert np.array_equal(_host(Zg2), _host(Zg)) and np.array_equal(_host(Rg2), _host(Rg)), "tdp_blend_cond"

    # mean over tiles, a length that is not a multiple of the vector width
    L = 8 * 37 + 8
    A = np.random.default_rng(wl.seed + 9).standard_normal((nt, B, L), dtype=np.float32)
    A = A if wl.dtype == "f32" else wk.f32_to_bf16_bits(A)
    Ag = _input(A)
    Mg = _output((B, L), lat)
    tdp.tdp_tile_mean(plan, L, Ag.t, Mg.t)
    torch.cuda.synchronize()
    _check_bands({"out": Mg}, "tdp_tile_mean")
    assert_blend_close(_host(Mg), oracle.tile_mean(p, A, L), wl)

    # inputs are never written either
    _check_bands({"X": Xg, "P": Pg, "K": Kg, "Yout": Yg, "Ycond": Ycg, "slot": Sg, "A": Ag}, "inputs")
    assert np.array_equal(_host(Xg), X) and np.array_equal(_host(Kg), K)
    plan.close()
