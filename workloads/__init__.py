"""Seeded synthetic inputs for the TDP tile split / blend workloads.

This module is shared by the tests, the benchmark and the smoke check.  It
holds shapes and random draws only -- none of the tiling arithmetic (tile
boxes, masks, offsets) -- so that neither the CPU oracle nor the CUDA path
can lean on the other through it.

Workloads (patchified video latent ``X[B,F,H,W,C]``, token positions
``P[B,3,T,2]`` with T = F*H*W, conditioning-token intervals ``K[B,3,N,2]``):

  tiny     B=1 F=3  H=8   W=12  C=16  fp32  tiles 1x2x2  overlap (0,2,2)  N=32    25% negative time
  small    B=1 F=16 H=32  W=48  C=128 bf16  tiles 1x2x2  overlap (0,8,8)  N=1024  10%
  medium   B=1 F=16 H=64  W=96  C=128 bf16  tiles 1x4x4  overlap (0,8,8)  N=4096   5%
  temporal B=2 F=32 H=68  W=120 C=128 bf16  tiles 2x3x3  overlap (4,8,8)  N=8192   5%
  large    B=1 F=64 H=128 W=192 C=128 bf16  tiles 2x8x8  overlap (4,16,16) N=16384 5%

Generated token positions are width-1 intervals on the latent grid:
start = (f, h, w), end = start + 1.  Conditioning tokens draw, per batch item
and per dimension, start ~ U{0..L-1} and end = start + U{1..max(1, L//4)};
a fixed fraction of them instead gets a negative time start ~ U{-8..-1} with
end = start + U{1..4}.  Tile outputs (the stand-in for the per-tile
transformer) are the split tile plus N(0, sigma) noise.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "by_name",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "make_latent",
    "make_gen_positions",
    "make_cond_positions",
    "make_noise",
    "make_inputs",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    F: int
    H: int
    W: int
    C: int
    dtype: str                 # "f32" or "bf16"
    num_tiles: tuple           # (n_F, n_H, n_W)
    overlap: tuple             # (o_F, o_H, o_W), latent grid units
    n_cond: int                # conditioning tokens per batch item
    neg_frac: float            # fraction of conditioning tokens with negative time
    sigma: float               # std of the stand-in transformer's output noise
    seed: int

    @property
    def dims(self):
        return (self.F, self.H, self.W)

    @property
    def tokens(self):
        return self.F * self.H * self.W

    @property
    def esize(self):
        return 4 if self.dtype == "f32" else 2

    def latent_bytes(self):
        return self.B * self.tokens * self.C * self.esize

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = [
    Workload("tiny", 1, 3, 8, 12, 16, "f32", (1, 2, 2), (0, 2, 2), 32, 0.25, 0.01, 1001),
    Workload("small", 1, 16, 32, 48, 128, "bf16", (1, 2, 2), (0, 8, 8), 1024, 0.10, 0.05, 1002),
    Workload("medium", 1, 16, 64, 96, 128, "bf16", (1, 4, 4), (0, 8, 8), 4096, 0.05, 0.05, 1003),
    Workload("temporal", 2, 32, 68, 120, 128, "bf16", (2, 3, 3), (4, 8, 8), 8192, 0.05, 0.05, 1004),
    Workload("large", 1, 64, 128, 192, 128, "bf16", (2, 8, 8), (4, 16, 16), 16384, 0.05, 0.05, 1005),
]


def by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


# --------------------------------------------------------------------------
# bf16 storage: numpy has no bfloat16, so bf16 tensors travel as uint16 bits.
# --------------------------------------------------------------------------
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    out = (u >> 16) & 1
    out += 0x7FFF
    out += u            # finite inputs only: wraps only for NaN/Inf bit patterns
    out >>= 16
    return out.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _store(a32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(a32, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(a32)
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------
def make_latent(wl: Workload, rng: np.random.Generator) -> np.ndarray:
    """X[B,F,H,W,C] ~ N(0,1) in the workload's storage type (uint16 bits for bf16)."""
    x = rng.standard_normal((wl.B, wl.F, wl.H, wl.W, wl.C), dtype=np.float32)
    return _store(x, wl.dtype)


def make_gen_positions(wl: Workload) -> np.ndarray:
    """P[B,3,T,2] int32: width-1 [start,end) intervals on the (F,H,W) grid, token order row-major."""
    f, h, w = np.meshgrid(np.arange(wl.F), np.arange(wl.H), np.arange(wl.W), indexing="ij")
    start = np.stack([f.ravel(), h.ravel(), w.ravel()]).astype(np.int32)   # [3,T]
    p = np.empty((wl.B, 3, wl.tokens, 2), dtype=np.int32)
    p[..., 0] = start[None]
    p[..., 1] = start[None] + 1
    return p


def make_cond_positions(wl: Workload, rng: np.random.Generator,
                        n_cond: Optional[int] = None,
                        edges: Optional[Sequence[Sequence[int]]] = None,
                        edge_frac: float = 0.0) -> np.ndarray:
    """K[B,3,N,2] int32 conditioning-token [start,end) intervals.

    ``edges`` (optional, one list of grid coordinates per dimension) lets a
    caller ask for intervals that end exactly on, or start just below, given
    coordinates: an ``edge_frac`` share of the non-negative tokens gets, in one
    random dimension, either end == e or start == e - 1 for a random e.
    """
    N = wl.n_cond if n_cond is None else n_cond
    L = wl.dims
    K = np.empty((wl.B, 3, N, 2), dtype=np.int32)
    n_neg = int(round(wl.neg_frac * N))
    for b in range(wl.B):
        for d in range(3):
            s = rng.integers(0, L[d], size=N)
            e = s + rng.integers(1, max(1, L[d] // 4) + 1, size=N)
            K[b, d, :, 0] = s
            K[b, d, :, 1] = e
        neg = rng.permutation(N)[:n_neg]
        s = rng.integers(-8, 0, size=n_neg)
        K[b, 0, neg, 0] = s
        K[b, 0, neg, 1] = s + rng.integers(1, 5, size=n_neg)
        if edges is not None and edge_frac > 0.0 and N > 0:
            pos = np.setdiff1d(np.arange(N), neg)
            n_edge = int(round(edge_frac * len(pos)))
            pick = rng.permutation(pos)[:n_edge]
            for k in pick:
                d = int(rng.integers(0, 3))
                cand = list(edges[d])
                if not cand:
                    continue
                e = int(cand[int(rng.integers(0, len(cand)))])
                width = int(rng.integers(1, max(1, L[d] // 4) + 1))
                if rng.integers(0, 2) == 0 and e - width >= 0:
                    K[b, d, k, 0], K[b, d, k, 1] = e - width, e          # ends on e
                elif e - 1 >= 0:
                    K[b, d, k, 0], K[b, d, k, 1] = e - 1, e - 1 + width  # starts at e-1
    return K


def make_noise(shape, sigma: float, rng: np.random.Generator) -> np.ndarray:
    """float32 N(0, sigma) noise of the given shape (the stand-in model's perturbation)."""
    return (sigma * rng.standard_normal(shape, dtype=np.float32)).astype(np.float32)


def make_inputs(wl: Workload):
    """(X, P, K) for a workload from its fixed seed."""
    rng = np.random.default_rng(wl.seed)
    X = make_latent(wl, rng)
    P = make_gen_positions(wl)
    K = make_cond_positions(wl, rng)
    return X, P, K
