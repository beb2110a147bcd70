"""GB300 Tiled Data Parallelism (TDP) tile split / blend -- Python binding.

A thin ctypes layer over ``libtdp.so`` (the C ABI in ``include/tdp.h``): the
functions here carry the C names, check that each torch tensor is a CUDA
tensor of the size, dtype and contiguity the plan implies (so a wrong buffer
is refused on the host instead of being overrun on the device), and pass raw
pointers and the current CUDA stream through.  Every step of the path runs in
the library's CUDA kernels; there is no fallback.  Importing this package
loads ``libtdp.so`` and raises if it has not been built
(``python blend_tdp_tile_gb300/build.py`` or ``__graft_entry__.build()``).

Method: "Tiled Data Parallelism (TDP)" (LTX-2 docs, multigpu) -- split a
patchified latent into overlapping (frames, height, width) tiles with their
positions ("What it is"), normalise each tile's positions ("Position
normalization"), filter conditioning tokens per tile ("Shared negative
(reference) positions"), and blend the tile outputs with trapezoidal masks
that sum to one ("What it is").
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "TDP_OK", "TDP_F32", "TDP_BF16", "TDP_MAX_TILES_PER_DIM", "TdpError",
    "Plan", "tdp_plan_create", "tdp_plan_info", "tdp_plan_destroy",
    "tdp_pos_bounds", "tdp_split", "tdp_split_tma", "tdp_norm_filter", "tdp_split_filter", "tdp_blend", "tdp_cond_blend",
    "tdp_cond_records_size", "tdp_cond_records", "tdp_cond_blend_records",
    "tdp_tile_mean", "tdp_blend_partial", "tdp_blend_store", "tdp_blend_cond",
    "tdp_balanced_tile_split", "tdp_tiles_for_size", "tdp_rank_tiles",
    "tdp_status_str", "tdp_last_error_detail",
    "alloc_split_outputs", "alloc_filter_outputs", "LIB_PATH",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtdp.so")

TDP_OK = 0
TDP_F32, TDP_BF16 = 0, 1
TDP_MAX_TILES_PER_DIM = 64


class TdpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tdp_status_str(status)} ({tdp_last_error_detail()})")


class _DimCfg(ctypes.Structure):
    _fields_ = [("num_tiles", ctypes.c_int32), ("overlap", ctypes.c_int32)]


class _Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("F", ctypes.c_int32), ("H", ctypes.c_int32),
                ("W", ctypes.c_int32), ("C", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("dim", _DimCfg * 3)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python blend_tdp_tile_gb300/build.py` or __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64p = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64)
    lib.tdp_plan_create.argtypes = [ctypes.POINTER(_Problem), ctypes.POINTER(vp)]
    lib.tdp_plan_create.restype = ctypes.c_int
    lib.tdp_plan_info.argtypes = [vp, ctypes.POINTER(i32), i64p, vp, vp]
    lib.tdp_plan_info.restype = ctypes.c_int
    lib.tdp_plan_destroy.argtypes = [vp]
    lib.tdp_plan_destroy.restype = None
    lib.tdp_pos_bounds.argtypes = [vp, vp, vp, vp, vp]
    lib.tdp_pos_bounds.restype = ctypes.c_int
    lib.tdp_split.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp]
    lib.tdp_split.restype = ctypes.c_int
    lib.tdp_split_tma.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp]
    lib.tdp_split_tma.restype = ctypes.c_int
    lib.tdp_norm_filter.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.tdp_norm_filter.restype = ctypes.c_int
    lib.tdp_split_filter.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.tdp_split_filter.restype = ctypes.c_int
    lib.tdp_cond_blend.argtypes = [vp, i32, i32, vp, vp, vp, vp]
    lib.tdp_cond_blend.restype = ctypes.c_int
    lib.tdp_cond_records_size.argtypes = [vp, i32, i64p]
    lib.tdp_cond_records_size.restype = ctypes.c_int
    lib.tdp_cond_records.argtypes = [vp, i32, i32, vp, vp, vp]
    lib.tdp_cond_records.restype = ctypes.c_int
    lib.tdp_cond_blend_records.argtypes = [vp, i32, i32, vp, vp, vp, vp]
    lib.tdp_cond_blend_records.restype = ctypes.c_int
    lib.tdp_tile_mean.argtypes = [vp, ctypes.c_int64, vp, vp, vp]
    lib.tdp_tile_mean.restype = ctypes.c_int
    lib.tdp_blend.argtypes = [vp, vp, vp, vp]
    lib.tdp_blend.restype = ctypes.c_int
    lib.tdp_blend_cond.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, vp]
    lib.tdp_blend_cond.restype = ctypes.c_int
    lib.tdp_blend_partial.argtypes = [vp, i32, i32, vp, vp, vp]
    lib.tdp_blend_partial.restype = ctypes.c_int
    lib.tdp_blend_store.argtypes = [vp, ctypes.c_int64, vp, vp, vp]
    lib.tdp_blend_store.restype = ctypes.c_int
    lib.tdp_balanced_tile_split.argtypes = [i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.tdp_balanced_tile_split.restype = ctypes.c_int
    lib.tdp_tiles_for_size.argtypes = [i32, i32, i32, ctypes.POINTER(i32)]
    lib.tdp_tiles_for_size.restype = ctypes.c_int
    lib.tdp_rank_tiles.argtypes = [vp, i32, i32, vp, ctypes.POINTER(i32)]
    lib.tdp_rank_tiles.restype = ctypes.c_int
    lib.tdp_status_str.argtypes = [ctypes.c_int]
    lib.tdp_status_str.restype = ctypes.c_char_p
    lib.tdp_last_error_detail.argtypes = []
    lib.tdp_last_error_detail.restype = ctypes.c_char_p
    return lib


_lib = _load()


def tdp_status_str(status: int) -> str:
    return _lib.tdp_status_str(int(status)).decode()


def tdp_last_error_detail() -> str:
    return _lib.tdp_last_error_detail().decode()


def _check(status: int, where: str):
    if status != TDP_OK:
        raise TdpError(status, where)


class Plan:
    """Owning wrapper of a ``tdp_plan_t``; geometry read back through tdp_plan_info."""

    def __init__(self, handle: int, problem: dict):
        self._h = ctypes.c_void_p(handle)
        self.problem = problem
        n = ctypes.c_int32()
        tot = ctypes.c_int64()
        _check(_lib.tdp_plan_info(self._h, ctypes.byref(n), ctypes.byref(tot), None, None), "tdp_plan_info")
        self.n_tiles = int(n.value)
        self.total_tile_tokens = int(tot.value)
        self.boxes = np.zeros((self.n_tiles, 3, 2), np.int32)
        self.offsets = np.zeros(self.n_tiles + 1, np.int64)
        _check(_lib.tdp_plan_info(self._h, None, None, self.boxes.ctypes.data_as(ctypes.c_void_p),
                                  self.offsets.ctypes.data_as(ctypes.c_void_p)), "tdp_plan_info")
        for k in ("B", "F", "H", "W", "C", "dtype"):
            setattr(self, k, problem[k])

    @property
    def handle(self):
        return self._h

    @property
    def esize(self):
        return 4 if self.dtype == TDP_F32 else 2

    def close(self):
        if self._h is not None and self._h.value:
            _lib.tdp_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tdp_plan_create(B, F, H, W, C, dtype, num_tiles, overlap) -> Plan:
    """Validate a problem and compute its tiles (host only).  dtype: TDP_F32/TDP_BF16 or 'f32'/'bf16'."""
    if isinstance(dtype, str):
        dtype = {"f32": TDP_F32, "bf16": TDP_BF16}[dtype]
    pr = _Problem()
    pr.B, pr.F, pr.H, pr.W, pr.C, pr.dtype = B, F, H, W, C, dtype
    for d in range(3):
        pr.dim[d].num_tiles = int(num_tiles[d])
        pr.dim[d].overlap = int(overlap[d])
    h = ctypes.c_void_p()
    _check(_lib.tdp_plan_create(ctypes.byref(pr), ctypes.byref(h)), "tdp_plan_create")
    return Plan(h.value, dict(B=B, F=F, H=H, W=W, C=C, dtype=dtype,
                              num_tiles=tuple(num_tiles), overlap=tuple(overlap)))


def tdp_plan_info(plan: Plan):
    """(n_tiles, total_tile_tokens, boxes[nt,3,2], offsets[nt+1])."""
    return plan.n_tiles, plan.total_tile_tokens, plan.boxes.copy(), plan.offsets.copy()


def tdp_plan_destroy(plan: Plan):
    plan.close()


def tdp_balanced_tile_split(world: int):
    """(h_tiles, w_tiles) for `world` ranks: the factor pair closest to square, h <= w."""
    h, w = ctypes.c_int32(), ctypes.c_int32()
    _check(_lib.tdp_balanced_tile_split(int(world), ctypes.byref(h), ctypes.byref(w)), "tdp_balanced_tile_split")
    return int(h.value), int(w.value)


def tdp_tiles_for_size(L: int, tile_size: int, overlap: int) -> int:
    """Smallest valid tile count along a dimension of extent L whose tiles fit in tile_size."""
    n = ctypes.c_int32()
    _check(_lib.tdp_tiles_for_size(int(L), int(tile_size), int(overlap), ctypes.byref(n)), "tdp_tiles_for_size")
    return int(n.value)


def tdp_rank_tiles(plan: Plan, rank: int, world: int) -> np.ndarray:
    """Tile ids rank `rank` of `world` runs under round-robin assignment (tile t -> t % world)."""
    tiles = np.zeros(max(plan.n_tiles, 1), np.int32)
    n = ctypes.c_int32()
    _check(_lib.tdp_rank_tiles(plan.handle, int(rank), int(world), tiles.ctypes.data_as(ctypes.c_void_p),
                               ctypes.byref(n)), "tdp_rank_tiles")
    return tiles[:n.value].copy()


# ------------------------------------------------------------------ marshalling
def _torch():
    import torch
    return torch


def _ptr(t, name, numel, dtypes, align):
    """Device pointer of a CUDA tensor after size/dtype/contiguity checks; None -> NULL."""
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")
    p = t.data_ptr()
    if p % align:
        raise ValueError(f"{name}: not {align}-byte aligned")
    return p


def _common_device(where, named):
    """The one device every given buffer lives on (None if no buffer is given).

    The library launches on the current CUDA device, so buffers of one call must share a
    device: a pointer of another device would reach the kernel as a foreign address.
    `named` holds (name, tensor-or-None) pairs; only `.device` of each is read."""
    dev, first = None, None
    for name, t in named:
        if t is None:
            continue
        if dev is None:
            dev, first = t.device, name
        elif t.device != dev:
            raise ValueError(f"{where}: {name} is on {t.device} but {first} is on {dev}")
    return dev


def _stream_handle(where, stream, dev):
    """Raw cudaStream_t for `stream` on device `dev`: None -> that device's current torch
    stream; a torch stream must belong to `dev`; an int is taken as a raw handle."""
    if stream is None:
        return _torch().cuda.current_stream(dev).cuda_stream
    if isinstance(stream, int):
        return stream
    sdev = getattr(stream, "device", None)
    if dev is not None and sdev is not None and sdev != dev:
        raise ValueError(f"{where}: stream is on {sdev} but the buffers are on {dev}")
    return stream.cuda_stream


class _Call:
    """Marshals one entry-point call: checks each buffer (size, dtype, contiguity,
    alignment, one common device), then calls the library with that device current."""

    def __init__(self, where):
        self.where = where
        self.named = []

    def ptr(self, t, name, numel, dtypes, align):
        p = _ptr(t, name, numel, dtypes, align)
        self.named.append((name, t))
        return p

    def run(self, fn, *args, stream=None):
        torch = _torch()
        dev = _common_device(self.where, self.named)
        if dev is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        with torch.cuda.device(dev):
            _check(fn(*args, _stream_handle(self.where, stream, dev)), self.where)


def _latent_dtypes(plan):
    torch = _torch()
    return (torch.float32,) if plan.dtype == TDP_F32 else (torch.bfloat16,)


def tdp_pos_bounds(plan: Plan, P, mn, mx, stream=None):
    """Every tile's min start / max end of its generated positions P [B,3,T,2] into mn, mx [nt,B,3]."""
    torch = _torch()
    B, T, nt = plan.B, plan.F * plan.H * plan.W, plan.n_tiles
    i32 = (torch.int32,)
    c = _Call("tdp_pos_bounds")
    c.run(_lib.tdp_pos_bounds, plan.handle, c.ptr(P, "P", B * 3 * T * 2, i32, 8),
          c.ptr(mn, "mn", nt * B * 3, i32, 4), c.ptr(mx, "mx", nt * B * 3, i32, 4), stream=stream)


def tdp_split(plan: Plan, X, P, mn, normalize, Y, Q, stream=None):
    """Split X [B,F,H,W,C] (and positions P [B,3,T,2], shifted by mn when normalising) into
    tile-major Y (and Q)."""
    torch = _torch()
    B, T, C, nt, tot = plan.B, plan.F * plan.H * plan.W, plan.C, plan.n_tiles, plan.total_tile_tokens
    lat = _latent_dtypes(plan)
    c = _Call("tdp_split")
    c.run(_lib.tdp_split, plan.handle,
          c.ptr(X, "X", B * T * C, lat, 16),
          c.ptr(P, "P", B * 3 * T * 2, (torch.int32,), 8),
          c.ptr(mn, "mn", nt * B * 3, (torch.int32,), 4),
          int(bool(normalize)),
          c.ptr(Y, "Y", B * tot * C, lat, 16),
          c.ptr(Q, "Q", B * tot * 6, (torch.int32,), 8), stream=stream)


def tdp_split_tma(plan: Plan, X, P, mn, normalize, Y, Q, err=None, stream=None):
    """tdp_split with the latent moved by bulk-tensor loads and bulk stores (same outputs);
    `err` (one int32 on the device, or None) is set to 1 if a load timed out."""
    torch = _torch()
    B, T, C, nt, tot = plan.B, plan.F * plan.H * plan.W, plan.C, plan.n_tiles, plan.total_tile_tokens
    lat = _latent_dtypes(plan)
    c = _Call("tdp_split_tma")
    c.run(_lib.tdp_split_tma, plan.handle,
          c.ptr(X, "X", B * T * C, lat, 16),
          c.ptr(P, "P", B * 3 * T * 2, (torch.int32,), 8),
          c.ptr(mn, "mn", nt * B * 3, (torch.int32,), 4),
          int(bool(normalize)),
          c.ptr(Y, "Y", B * tot * C, lat, 16),
          c.ptr(Q, "Q", B * tot * 6, (torch.int32,), 8),
          c.ptr(err, "err", 1, (torch.int32,), 4), stream=stream)


def tdp_norm_filter(plan: Plan, K, N, mn, mx, normalize, keep, idx, count, kcount, Kout, slot=None,
                    stream=None):
    """Per-tile keep / compaction / normalisation of conditioning tokens K [B,3,N,2]
    (and, if `slot` is given, each token's position in every tile's kept list)."""
    torch = _torch()
    B, nt = plan.B, plan.n_tiles
    N = int(N)
    i32 = (torch.int32,)
    c = _Call("tdp_norm_filter")
    c.run(_lib.tdp_norm_filter, plan.handle,
          c.ptr(K, "K", B * 3 * N * 2, i32, 8), N,
          c.ptr(mn, "mn", nt * B * 3, i32, 4),
          c.ptr(mx, "mx", nt * B * 3, i32, 4),
          int(bool(normalize)),
          c.ptr(keep, "keep", nt * B * N, (torch.uint8,), 1),
          c.ptr(idx, "idx", nt * B * N, i32, 4),
          c.ptr(count, "count", nt * B, i32, 4),
          c.ptr(kcount, "kcount", B * N, i32, 4),
          c.ptr(Kout, "Kout", nt * B * 3 * N * 2, i32, 8),
          c.ptr(slot, "slot", nt * B * N, i32, 4), stream=stream)


def tdp_split_filter(plan: Plan, X, P, K, N, normalize, Y, Q, mn, mx, keep, idx, count, kcount, Kout,
                     slot=None, stream=None):
    """tdp_pos_bounds + tdp_split + tdp_norm_filter in one call (three launches): the same
    outputs, bit for bit."""
    torch = _torch()
    B, T, C, nt, tot = plan.B, plan.F * plan.H * plan.W, plan.C, plan.n_tiles, plan.total_tile_tokens
    N = int(N)
    lat = _latent_dtypes(plan)
    i32 = (torch.int32,)
    c = _Call("tdp_split_filter")
    c.run(_lib.tdp_split_filter, plan.handle,
          c.ptr(X, "X", B * T * C, lat, 16),
          c.ptr(P, "P", B * 3 * T * 2, i32, 8),
          c.ptr(K, "K", B * 3 * N * 2, i32, 8), N,
          int(bool(normalize)),
          c.ptr(Y, "Y", B * tot * C, lat, 16),
          c.ptr(Q, "Q", B * tot * 6, i32, 8),
          c.ptr(mn, "mn", nt * B * 3, i32, 4),
          c.ptr(mx, "mx", nt * B * 3, i32, 4),
          c.ptr(keep, "keep", nt * B * N, (torch.uint8,), 1),
          c.ptr(idx, "idx", nt * B * N, i32, 4),
          c.ptr(count, "count", nt * B, i32, 4),
          c.ptr(kcount, "kcount", B * N, i32, 4),
          c.ptr(Kout, "Kout", nt * B * 3 * N * 2, i32, 8),
          c.ptr(slot, "slot", nt * B * N, i32, 4), stream=stream)


def tdp_cond_blend(plan: Plan, N, ncap, Ycond, slot, out, stream=None):
    """Average each conditioning token's per-tile outputs Ycond [nt,B,ncap,C] over the tiles
    that kept it (slot from tdp_norm_filter) into out [B,N,C]."""
    torch = _torch()
    B, nt, C = plan.B, plan.n_tiles, plan.C
    N, ncap = int(N), int(ncap)
    lat = _latent_dtypes(plan)
    c = _Call("tdp_cond_blend")
    c.run(_lib.tdp_cond_blend, plan.handle, N, ncap, c.ptr(Ycond, "Ycond", nt * B * ncap * C, lat, 16),
          c.ptr(slot, "slot", nt * B * N, (torch.int32,), 4),
          c.ptr(out, "out", B * N * C, lat, 16), stream=stream)


def tdp_cond_records_size(plan: Plan, N) -> int:
    """int32 elements of the records tdp_cond_records writes for N conditioning tokens."""
    n = ctypes.c_int64(0)
    _check(_lib.tdp_cond_records_size(plan.handle, int(N), ctypes.byref(n)), "tdp_cond_records_size")
    return n.value


def tdp_cond_records(plan: Plan, N, ncap, slot, recs, stream=None):
    """Once per set of conditioning tokens: the tokens dealt to records of 8 by stored rows, and
    every record (its tokens, their rows and weights), into recs (int32,
    tdp_cond_records_size elements)."""
    torch = _torch()
    B, nt, N, ncap = plan.B, plan.n_tiles, int(N), int(ncap)
    c = _Call("tdp_cond_records")
    c.run(_lib.tdp_cond_records, plan.handle, N, ncap, c.ptr(slot, "slot", nt * B * N, (torch.int32,), 4),
          c.ptr(recs, "recs", tdp_cond_records_size(plan, N), (torch.int32,), 16), stream=stream)


def tdp_cond_blend_records(plan: Plan, N, recs, Ycond, ncap, out, stream=None):
    """tdp_cond_blend from the records tdp_cond_records made (same plan, N, ncap and slot)."""
    torch = _torch()
    B, nt, C, N, ncap = plan.B, plan.n_tiles, plan.C, int(N), int(ncap)
    lat = _latent_dtypes(plan)
    c = _Call("tdp_cond_blend_records")
    c.run(_lib.tdp_cond_blend_records, plan.handle, N, ncap,
          c.ptr(recs, "recs", tdp_cond_records_size(plan, N), (torch.int32,), 16),
          c.ptr(Ycond, "Ycond", nt * B * ncap * C, lat, 16), c.ptr(out, "out", B * N * C, lat, 16), stream=stream)


def tdp_tile_mean(plan: Plan, L, A, out, stream=None):
    """Mean over tiles of A [nt,B,L] into out [B,L] (the audio path)."""
    B, nt, L = plan.B, plan.n_tiles, int(L)
    lat = _latent_dtypes(plan)
    c = _Call("tdp_tile_mean")
    c.run(_lib.tdp_tile_mean, plan.handle, L, c.ptr(A, "A", nt * B * L, lat, 16),
          c.ptr(out, "out", B * L, lat, 16), stream=stream)


def tdp_blend(plan: Plan, Yout, Z, stream=None):
    """Blend tile-major tile outputs Yout into Z [B,F,H,W,C] with the trapezoidal masks."""
    B, T, C, tot = plan.B, plan.F * plan.H * plan.W, plan.C, plan.total_tile_tokens
    lat = _latent_dtypes(plan)
    c = _Call("tdp_blend")
    c.run(_lib.tdp_blend, plan.handle, c.ptr(Yout, "Yout", B * tot * C, lat, 16),
          c.ptr(Z, "Z", B * T * C, lat, 16), stream=stream)


def tdp_blend_cond(plan: Plan, Yout, Z, N, ncap, Ycond, slot, out, stream=None):
    """tdp_blend (Yout -> Z) and tdp_cond_blend (Ycond, slot -> out) in one call (one launch):
    the same outputs, bit for bit."""
    torch = _torch()
    B, T, C, nt, tot = plan.B, plan.F * plan.H * plan.W, plan.C, plan.n_tiles, plan.total_tile_tokens
    N, ncap = int(N), int(ncap)
    lat = _latent_dtypes(plan)
    c = _Call("tdp_blend_cond")
    c.run(_lib.tdp_blend_cond, plan.handle, c.ptr(Yout, "Yout", B * tot * C, lat, 16),
          c.ptr(Z, "Z", B * T * C, lat, 16), N, ncap,
          c.ptr(Ycond, "Ycond", nt * B * ncap * C, lat, 16),
          c.ptr(slot, "slot", nt * B * N, (torch.int32,), 4),
          c.ptr(out, "out", B * N * C, lat, 16), stream=stream)


def tdp_blend_partial(plan: Plan, rank, world, Yout, Zp, stream=None):
    """Rank `rank` of `world`'s share of the blend (its round-robin tiles t % world == rank)
    into the fp32 partial latent Zp [B,F,H,W,C]."""
    torch = _torch()
    B, T, C, tot = plan.B, plan.F * plan.H * plan.W, plan.C, plan.total_tile_tokens
    lat = _latent_dtypes(plan)
    c = _Call("tdp_blend_partial")
    c.run(_lib.tdp_blend_partial, plan.handle, int(rank), int(world), c.ptr(Yout, "Yout", B * tot * C, lat, 16),
          c.ptr(Zp, "Zp", B * T * C, (torch.float32,), 16), stream=stream)


def tdp_blend_store(plan: Plan, Zsum, Z, stream=None):
    """Z = Zsum (fp32) in the plan's dtype; Zsum and Z have the same number of elements (the
    whole latent or a run of whole rows)."""
    torch = _torch()
    n = int(Zsum.numel())
    lat = _latent_dtypes(plan)
    c = _Call("tdp_blend_store")
    c.run(_lib.tdp_blend_store, plan.handle, n, c.ptr(Zsum, "Zsum", n, (torch.float32,), 16),
          c.ptr(Z, "Z", n, lat, 16), stream=stream)


# ------------------------------------------------------------------ allocation helpers
def alloc_split_outputs(plan: Plan, device="cuda", positions=True):
    """Y [B*total, C], Q [B*total*6], mn, mx [nt,B,3] on `device` (torch allocations)."""
    torch = _torch()
    dt = torch.float32 if plan.dtype == TDP_F32 else torch.bfloat16
    Y = torch.empty((plan.B * plan.total_tile_tokens, plan.C), dtype=dt, device=device)
    if not positions:
        return Y, None, None, None
    Q = torch.empty(plan.B * plan.total_tile_tokens * 6, dtype=torch.int32, device=device)
    mn = torch.empty((plan.n_tiles, plan.B, 3), dtype=torch.int32, device=device)
    mx = torch.empty_like(mn)
    return Y, Q, mn, mx


def alloc_filter_outputs(plan: Plan, N: int, device="cuda", slot=False):
    """keep, idx [nt,B,N], count [nt,B], kcount [B,N], Kout [nt,B,3,N,2] (and slot [nt,B,N])."""
    torch = _torch()
    nt, B = plan.n_tiles, plan.B
    keep = torch.empty((nt, B, N), dtype=torch.uint8, device=device)
    idx = torch.empty((nt, B, N), dtype=torch.int32, device=device)
    count = torch.empty((nt, B), dtype=torch.int32, device=device)
    kcount = torch.empty((B, N), dtype=torch.int32, device=device)
    Kout = torch.empty((nt, B, 3, N, 2), dtype=torch.int32, device=device)
    if slot:
        return keep, idx, count, kcount, Kout, torch.empty((nt, B, N), dtype=torch.int32, device=device)
    return keep, idx, count, kcount, Kout
