"""CPU oracle for the TDP tile split / normalisation / filter / blend.

TEST INFRASTRUCTURE ONLY.  This package is the checker the CUDA library is
compared against: the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg are the only code that may import it.  It shares no code
with ``blend_tdp_tile_gb300`` and never imports it.

The arithmetic lives in ``tdp_oracle.c`` (plain C loops, fp64 blend); this
module compiles it with gcc on first use and marshals numpy arrays through
ctypes.  Every function follows "Tiled Data Parallelism (TDP)" (LTX-2 docs,
multigpu); the C file names the section each step restates and the reading
taken where the page is silent.

Parity pins (checked by the CPU test-suite against facts that do not come
from this code): the tiny workload's 3x5x7 tile size, exact integer partition
of unity of the ramps, linear ramps, split == numpy box slicing, identity for
one tile, pure permutation for zero overlap, blend(split(X)) == X, closed-form
offsets for grid positions, negative-time tokens kept by every tile, cell
enumeration for the keep rule, an exact-rational brute force of the blend,
and, for the conditioning-output average and the audio tile mean, identity
outputs, per-tile constants, single-keeper tokens and one-tile copies.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tdp_oracle.c")
_DEFAULT_LIB = os.path.join(_HERE, "liboracle.so")
# Test hook: point the wrapper at another build of tdp_oracle.c (the mutation tests
# load deliberately broken copies to check that the pins catch them).
_LIB = os.environ.get("TDP_ORACLE_LIB") or _DEFAULT_LIB
_lock = threading.Lock()
_lib = None


class Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("F", ctypes.c_int32), ("H", ctypes.c_int32),
        ("W", ctypes.c_int32), ("C", ctypes.c_int32), ("esize", ctypes.c_int32),
        ("n", ctypes.c_int32 * 3), ("o", ctypes.c_int32 * 3),
    ]


def compile_source(src: str, out: str) -> str:
    """gcc -O2 -std=c11 -shared: one oracle source file into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, src])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile tdp_oracle.c into liboracle.so beside it (gcc, C11, -O2)."""
    if _LIB != _DEFAULT_LIB:
        return _LIB
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.POINTER(Problem)
            vp = ctypes.c_void_p
            i32 = ctypes.c_int32
            lib.oracle_tile_boxes_1d.argtypes = [i32, i32, i32, vp, vp]
            lib.oracle_tile_boxes_1d.restype = ctypes.c_int
            lib.oracle_num_tiles.argtypes = [P]
            lib.oracle_plan.argtypes = [P, vp, vp]
            lib.oracle_plan.restype = ctypes.c_int
            lib.oracle_ramp_num.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(i32)]
            lib.oracle_ramp_num.restype = i32
            lib.oracle_mask.argtypes = [P, i32, i32, i32, i32]
            lib.oracle_mask.restype = ctypes.c_double
            lib.oracle_split.argtypes = [P, vp, vp, vp, vp]
            lib.oracle_split.restype = None
            lib.oracle_bounds.argtypes = [P, vp, vp, vp]
            lib.oracle_bounds.restype = None
            lib.oracle_normalize.argtypes = [P, vp, vp]
            lib.oracle_normalize.restype = None
            lib.oracle_filter.argtypes = [P, vp, i32, vp, vp, i32, vp, vp, vp, vp, vp, vp]
            lib.oracle_filter.restype = None
            lib.oracle_blend.argtypes = [P, vp, vp]
            lib.oracle_blend.restype = None
            lib.oracle_blend_cell.argtypes = [P, vp, i32, i32, i32, i32, vp]
            lib.oracle_blend_cell.restype = None
            lib.oracle_cond_blend.argtypes = [P, i32, i32, vp, vp, vp, vp, vp]
            lib.oracle_cond_blend.restype = None
            lib.oracle_tile_mean.argtypes = [P, vp, ctypes.c_int64, vp]
            lib.oracle_tile_mean.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def problem(B, F, H, W, C, esize, num_tiles, overlap) -> Problem:
    p = Problem()
    p.B, p.F, p.H, p.W, p.C, p.esize = B, F, H, W, C, esize
    for d in range(3):
        p.n[d] = num_tiles[d]
        p.o[d] = overlap[d]
    return p


def problem_of(wl) -> Problem:
    """Problem for a ``workloads.Workload`` (or anything with the same fields)."""
    return problem(wl.B, wl.F, wl.H, wl.W, wl.C, wl.esize, wl.num_tiles, wl.overlap)


def tile_boxes_1d(L, n, o):
    lo = np.zeros(max(n, 1), np.int32)
    hi = np.zeros(max(n, 1), np.int32)
    rc = _load().oracle_tile_boxes_1d(L, n, o, _ptr(lo), _ptr(hi))
    if rc != 0:
        raise ValueError(f"invalid tiling L={L} n={n} o={o}")
    return lo, hi


def plan(p: Problem):
    """(box[nt,3,2] int32, off[nt+1] int64)."""
    lib = _load()
    nt = p.n[0] * p.n[1] * p.n[2]
    box = np.zeros((nt, 3, 2), np.int32)
    off = np.zeros(nt + 1, np.int64)
    if lib.oracle_plan(ctypes.byref(p), _ptr(box), _ptr(off)) != 0:
        raise ValueError("invalid tiling")
    return box, off


def ramp_num(L, n, o, i, x):
    """(numerator, denominator) of tile i's 1-D ramp at coordinate x."""
    den = ctypes.c_int32()
    num = _load().oracle_ramp_num(L, n, o, i, x, ctypes.byref(den))
    return int(num), int(den.value)


def mask(p: Problem, t, f, h, w) -> float:
    return float(_load().oracle_mask(ctypes.byref(p), t, f, h, w))


def _elem_dtype(p: Problem):
    return np.float32 if p.esize == 4 else np.uint16


def split(p: Problem, X: np.ndarray, P: np.ndarray):
    """(Y tile-major [B*sum T_t, C], Q tile-major [B*3*sum T_t*2]) -- see tdp_oracle.c."""
    box, off = plan(p)
    tot = int(off[-1])
    X = np.ascontiguousarray(X, dtype=_elem_dtype(p))
    P = np.ascontiguousarray(P, dtype=np.int32)
    Y = np.zeros((p.B * tot, p.C), _elem_dtype(p))
    Q = np.zeros(p.B * 3 * tot * 2, np.int32)
    _load().oracle_split(ctypes.byref(p), _ptr(X), _ptr(P), _ptr(Y), _ptr(Q))
    return Y, Q


def bounds(p: Problem, Q: np.ndarray):
    nt = p.n[0] * p.n[1] * p.n[2]
    Q = np.ascontiguousarray(Q, dtype=np.int32)
    mn = np.zeros((nt, p.B, 3), np.int32)
    mx = np.zeros((nt, p.B, 3), np.int32)
    _load().oracle_bounds(ctypes.byref(p), _ptr(Q), _ptr(mn), _ptr(mx))
    return mn, mx


def normalize(p: Problem, Q: np.ndarray, mn: np.ndarray) -> np.ndarray:
    Qn = np.array(Q, dtype=np.int32, copy=True, order="C")
    _load().oracle_normalize(ctypes.byref(p), _ptr(Qn), _ptr(np.ascontiguousarray(mn, np.int32)))
    return Qn


def filter_cond(p: Problem, K: np.ndarray, mn, mx, normalize_positions: bool = True, with_slot: bool = False):
    """(keep[nt,B,N] u8, idx[nt,B,N], count[nt,B], kcount[B,N], Kout[nt,B,3,N,2]) and, with
    `with_slot`, slot[nt,B,N] (token k's position in (t,b)'s kept list, or -1)."""
    nt = p.n[0] * p.n[1] * p.n[2]
    K = np.ascontiguousarray(K, dtype=np.int32)
    N = K.shape[2]
    keep = np.zeros((nt, p.B, N), np.uint8)
    idx = np.zeros((nt, p.B, N), np.int32)
    count = np.zeros((nt, p.B), np.int32)
    kcount = np.zeros((p.B, N), np.int32)
    Kout = np.zeros((nt, p.B, 3, N, 2), np.int32)
    slot = np.zeros((nt, p.B, N), np.int32)
    _load().oracle_filter(ctypes.byref(p), _ptr(K), N,
                          _ptr(np.ascontiguousarray(mn, np.int32)), _ptr(np.ascontiguousarray(mx, np.int32)),
                          int(bool(normalize_positions)),
                          _ptr(keep), _ptr(idx), _ptr(count), _ptr(kcount), _ptr(Kout), _ptr(slot))
    if with_slot:
        return keep, idx, count, kcount, Kout, slot
    return keep, idx, count, kcount, Kout


def cond_blend(p: Problem, Ycond: np.ndarray, keep, idx, count, ncap: int) -> np.ndarray:
    """out[B,N,C] float64: each conditioning token's outputs averaged over the tiles that kept it."""
    N = keep.shape[2]
    Ycond = np.ascontiguousarray(Ycond, dtype=_elem_dtype(p))
    out = np.zeros((p.B, N, p.C), np.float64)
    _load().oracle_cond_blend(ctypes.byref(p), N, ncap, _ptr(Ycond),
                              _ptr(np.ascontiguousarray(keep, np.uint8)),
                              _ptr(np.ascontiguousarray(idx, np.int32)),
                              _ptr(np.ascontiguousarray(count, np.int32)), _ptr(out))
    return out


def tile_mean(p: Problem, A: np.ndarray, L: int) -> np.ndarray:
    """out[B,L] float64: mean over tiles of A[nt,B,L]."""
    A = np.ascontiguousarray(A, dtype=_elem_dtype(p))
    out = np.zeros((p.B, L), np.float64)
    _load().oracle_tile_mean(ctypes.byref(p), _ptr(A), L, _ptr(out))
    return out


def blend(p: Problem, Yout: np.ndarray) -> np.ndarray:
    """Z[B,F,H,W,C] float64."""
    Yout = np.ascontiguousarray(Yout, dtype=_elem_dtype(p))
    Z = np.zeros((p.B, p.F, p.H, p.W, p.C), np.float64)
    _load().oracle_blend(ctypes.byref(p), _ptr(Yout), _ptr(Z))
    return Z


def blend_cell(p: Problem, Yout: np.ndarray, b, f, h, w) -> np.ndarray:
    Yout = np.ascontiguousarray(Yout, dtype=_elem_dtype(p))
    z = np.zeros(p.C, np.float64)
    _load().oracle_blend_cell(ctypes.byref(p), _ptr(Yout), b, f, h, w, _ptr(z))
    return z


def run_path(p: Problem, X, P, K, Yout=None, normalize_positions=True):
    """Whole hot path on the CPU: split -> bounds -> normalise -> filter -> blend.

    ``Yout`` defaults to the split tiles themselves (identity stand-in model).
    Returns a dict of every intermediate.
    """
    Y, Q = split(p, X, P)
    mn, mx = bounds(p, Q)
    Qn = normalize(p, Q, mn) if normalize_positions else Q
    keep, idx, count, kcount, Kout = filter_cond(p, K, mn, mx, normalize_positions)
    Z = blend(p, Y if Yout is None else Yout)
    return dict(Y=Y, Q=Qn, mn=mn, mx=mx, keep=keep, idx=idx, count=count,
                kcount=kcount, Kout=Kout, Z=Z)
