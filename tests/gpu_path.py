"""Helpers for the GPU parity tests: run the CUDA path through the binding on
numpy inputs and bring every output back to the host."""
from __future__ import annotations

import numpy as np


def torch_dtype(wl):
    import torch
    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def to_dev(a: np.ndarray, wl=None, dev="cuda"):
    """numpy -> CUDA tensor; uint16 arrays carry bf16 bits."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def to_host(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def fill_sentinel(t):
    """Pre-fill an output with a pattern no correct kernel writes everywhere."""
    import torch
    if t.dtype in (torch.float32, torch.bfloat16):
        t.fill_(float("nan"))
    elif t.dtype == torch.uint8:
        t.fill_(0xAB)
    else:
        t.fill_(-12345)
    return t


def run_split_filter(tdp, plan, wl, X, P, K, normalize=True, stream=None, positions=True, fused=False):
    """Bounds, split and filter on the GPU, every output pre-filled with a sentinel.
    fused=False: tdp_pos_bounds + tdp_split + tdp_norm_filter; fused=True: tdp_split_filter."""
    import torch
    dev = "cuda"
    Xd = to_dev(X)
    Pd = to_dev(P) if positions else None
    Y, Q, mn, mx = tdp.alloc_split_outputs(plan, dev, positions=positions)
    for t in (Y, Q, mn, mx):
        if t is not None:
            fill_sentinel(t)
    N = K.shape[2]
    if positions:
        keep, idx, count, kcount, Kout, slot = tdp.alloc_filter_outputs(plan, N, dev, slot=True)
        for t in (keep, idx, count, kcount, Kout, slot):
            fill_sentinel(t)
    if fused:
        assert positions
        tdp.tdp_split_filter(plan, Xd, Pd, to_dev(K), N, normalize, Y, Q, mn, mx, keep, idx, count, kcount,
                             Kout, slot, stream=stream)
    else:
        if positions:
            tdp.tdp_pos_bounds(plan, Pd, mn, mx, stream=stream)
        tdp.tdp_split(plan, Xd, Pd, mn, normalize, Y, Q, stream=stream)
        if positions:
            tdp.tdp_norm_filter(plan, to_dev(K), N, mn, mx, normalize, keep, idx, count, kcount, Kout,
                                slot, stream=stream)
    if stream is not None:
        stream.synchronize()
    torch.cuda.synchronize()
    out = dict(Yd=Y, Y=to_host(Y))
    if positions:
        out.update(Q=to_host(Q), mn=to_host(mn), mx=to_host(mx))
        out.update(keep=to_host(keep), idx=to_host(idx), count=to_host(count),
                   kcount=to_host(kcount), Kout=to_host(Kout), slot=to_host(slot), slotd=slot)
    return out


def run_blend(tdp, plan, wl, Yout, stream=None):
    import torch
    Yd = Yout if isinstance(Yout, torch.Tensor) else to_dev(Yout)
    Z = torch.empty((wl.B, wl.F, wl.H, wl.W, wl.C), dtype=torch_dtype(wl), device="cuda")
    fill_sentinel(Z)
    tdp.tdp_blend(plan, Yd, Z, stream=stream)
    if stream is not None:
        stream.synchronize()
    torch.cuda.synchronize()
    return Z


def as_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def blend_tolerance(wl):
    """Allowed |z - z*| per element against the fp64 oracle.

    bf16 storage: 2e-3 + 1e-2*|z*| (bf16 rounds to 2^-9 relative; fp32 weights and
    accumulation add ~1e-6).  fp32 storage: at most 8 terms with fp32 weights
    (3 roundings each) and fp32 accumulation: 1e-5 + 1e-5*|z*| bounds it with margin.
    """
    return (2e-3, 1e-2) if wl.dtype == "bf16" else (1e-5, 1e-5)


def assert_blend_close(z: np.ndarray, ref: np.ndarray, wl):
    atol, rtol = blend_tolerance(wl)
    z = as_f64(z)
    assert np.isfinite(z).all(), "blend left unwritten (NaN) elements"
    err = np.abs(z - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{int(bad.sum())} elements out of tolerance; max err {err.max():.3e}"


def assert_filter_equal(out, ref, nt, B):
    assert np.array_equal(out["keep"], ref["keep"])
    if "slot" in ref and "slot" in out:
        assert np.array_equal(out["slot"], ref["slot"])
    assert np.array_equal(out["idx"], ref["idx"])
    assert np.array_equal(out["count"], ref["count"])
    assert np.array_equal(out["kcount"], ref["kcount"])
    for t in range(nt):
        for b in range(B):
            c = ref["count"][t, b]
            assert np.array_equal(out["Kout"][t, b, :, :c], ref["Kout"][t, b, :, :c])
