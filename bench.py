#!/usr/bin/env python
"""Benchmark of the TDP hot path: tile split (+positions) -> conditioning filter -> blend.

One step = the pre-model stage (position bounds, tile split with normalised
positions, conditioning filter) and the blend over the large workload (B=1,
F=64, H=128, W=192, C=128 bf16; 2x8x8 tiles with overlap (4,16,16); 16384
conditioning tokens), inputs resident in HBM.  --path fused (default) runs the
pre-model stage as one tdp_split_filter call; --path separate as tdp_pos_bounds,
tdp_split and tdp_norm_filter.  The tile outputs fed to
the blend are the split tiles plus N(0, 0.05) noise, made once before timing
(the stand-in for the per-tile transformer, which is not part of the path).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  With torchrun (N > 1) every rank runs an independent
replica of the step (the path has no exchange on one GPU); the value is the
bytes of all ranks over the slowest rank's time.  --impl reference times the
CPU oracle on this host instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wk  # noqa: E402

METRIC = "TDP split+blend effective GB/s (fraction of GB300 HBM peak); latent tokens/s"
WORKLOAD = "large"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0     # GB300 HBM3e, nominal (context beside the measured peak)
AUDIO_TOKENS = 2048          # synthetic per-tile audio latent for the tile-mean timing
# kernels one step launches
LAUNCHES_PER_STEP = {
    "fused": 4,       # bounds init, bounds, split + filter, blend
    "separate": 6,    # bounds init, bounds, split, keep, compact, blend
}
# ncu DRAM-traffic summaries, one per workload: profiles/dram_traffic_<workload>.txt
PROFILE_DIR = os.path.join(ROOT, "profiles")
INSTRUMENT_EVERY = 10        # steps between those timed call by call


# ----------------------------------------------------------------------------- bytes
def algorithmic_bytes(wl, total_tile_tokens, n_tiles, kept_total=None):
    """Bytes each call must move at minimum (per batch of the workload).

    bounds: read the positions once, write mn / mx                 (B*T*24 + 2*nt*B*12)
    split : read the latent and positions once, write every tile token and its
            positions                                               (B*T*(C*e + 24) + B*sumT*(C*e + 24))
    filter: read cond tokens once, write keep/idx/kcount/count and the kept intervals
    blend : read every tile-output token once, write the latent     (B*sumT*C*e + B*T*C*e)
    The step counts the positions once (the bounds pass re-reads what the split reads).
    """
    B, T, C, e = wl.B, wl.tokens, wl.C, wl.esize
    tot = total_tile_tokens
    N = wl.n_cond
    mnmx = 2 * n_tiles * B * 3 * 4
    bounds = B * T * 24 + mnmx
    split = B * T * C * e + B * tot * C * e + B * T * 24 + B * tot * 24
    kept = kept_total if kept_total is not None else 0
    filt = B * N * 24 + n_tiles * B * N * (1 + 4) + n_tiles * B * 4 + B * N * 4 + kept * 24
    blend = B * tot * C * e + B * T * C * e
    return dict(bounds=bounds, split=split, filter=filt, blend=blend, step=mnmx + split + filt + blend)


L2_BYTES = 129 << 20          # GB300 L2


def config_of(wl, plan_tokens, n_tiles, parallelism, device=True):
    tile_bytes = wl.B * plan_tokens * wl.C * wl.esize
    lat_bytes = wl.latent_bytes()
    sizes = f"tile outputs {tile_bytes / 1e9:.2f} GB, latent {lat_bytes / 1e9:.2f} GB per step"
    if not device:
        l2 = f"host CPU ({sizes})"
    elif tile_bytes > L2_BYTES:
        l2 = f"inputs larger than L2 ({sizes}); no flush"
    else:
        l2 = f"inputs fit in L2 ({sizes}): not an HBM measurement"
    return {
        "workload": (f"{wl.name}: B={wl.B} F={wl.F} H={wl.H} W={wl.W} C={wl.C} {wl.dtype}, "
                     f"tiles {'x'.join(map(str, wl.num_tiles))}, overlap {tuple(wl.overlap)}, "
                     f"{n_tiles} tiles / {plan_tokens} tile tokens, {wl.n_cond} cond tokens"),
        "parallelism": parallelism,
        "l2": l2,
    }


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms (read-only query) while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.1 <= r[0] <= t1 + 0.1]
        note = "samples inside the timed region"
        if not inside:
            inside, note = rows, "timed region shorter than the sampling period: samples of the whole run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "note": note}


def gpu_id_for_smi(torch, dev):
    """nvidia-smi id (UUID when it can be matched) of the torch device."""
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        out = subprocess.run(["nvidia-smi", "--query-gpu=index,uuid", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            idx, u = [p.strip() for p in line.split(",")]
            if uuid and (u.endswith(uuid) or uuid.endswith(u.replace("GPU-", ""))):
                return u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    first = vis.split(",")[dev] if vis else str(dev)
    return first.strip() or "0"


# ----------------------------------------------------------------------------- peaks / traffic
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "blend_tdp_tile_gb300", "csrc", n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


_COMMON = ["tdp_device.cuh", "tdp_geom.h", "tdp_internal.h"]
KERNEL_SOURCES = {
    "tdp_blend_kernel": ["tdp_blend.cu"] + _COMMON,
    "tdp_split_kernel": ["tdp_split.cu", "tdp_filter.cuh"] + _COMMON,
    "tdp_split_filter_kernel": ["tdp_split.cu", "tdp_filter.cuh"] + _COMMON,
    "tdp_bounds_init_kernel": ["tdp_bounds.cu"] + _COMMON,
    "tdp_bounds_kernel": ["tdp_bounds.cu"] + _COMMON,
}
# the kernels each timed call launches
CALL_KERNELS = {
    "tdp_split_filter": ["tdp_bounds_init_kernel", "tdp_bounds_kernel", "tdp_split_filter_kernel"],
    "tdp_split": ["tdp_split_kernel"],
    "tdp_blend": ["tdp_blend_kernel"],
}


def profiled_traffic(call, workload=WORKLOAD):
    """DRAM bytes (read + write) of one `call` on `workload`, summed over its kernels, from
    the committed ncu summary of that workload; None when none was taken for it, or when a
    kernel's sources changed since the capture."""
    rows = {}
    try:
        with open(os.path.join(PROFILE_DIR, f"dram_traffic_{workload}.txt")) as fh:
            for line in fh:
                parts = line.split()
                if parts and not line.startswith("#"):
                    rows[parts[0]] = parts
        total = 0
        for k in CALL_KERNELS[call]:
            parts = rows[k]
            if parts[1] != kernel_source_hash(KERNEL_SOURCES[k]):
                return None
            total += int(parts[2]) + int(parts[3])
        return total
    except (OSError, ValueError, IndexError, KeyError):
        return None


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(x: float, device) -> float:
    """The largest `x` over all ranks of the default process group (every rank calls it)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle
def oracle_step_time(wl, X, P, K):
    """Wall time of one oracle pass (split, bounds, normalise, filter, blend) on one core."""
    import oracle
    p = oracle.problem_of(wl)
    t = time.perf_counter()
    Y, Q = oracle.split(p, X, P)
    mn, mx = oracle.bounds(p, Q)
    oracle.normalize(p, Q, mn)
    keep, idx, count, kcount, Kout = oracle.filter_cond(p, K, mn, mx, True)
    oracle.blend(p, Y)
    return time.perf_counter() - t, int(count.sum())


def cpu_baseline(wl, X, P, K, min_seconds=10.0, max_reps=20):
    import oracle
    oracle.build()
    box, off = oracle.plan(oracle.problem_of(wl))
    times, kept = [], 0
    while (sum(times) < min_seconds and len(times) < max_reps) or not times:
        dt, kept = oracle_step_time(wl, X, P, K)
        times.append(dt)
    ab = algorithmic_bytes(wl, int(off[-1]), box.shape[0], kept)["step"]
    mean = sum(times) / len(times)
    return {"value": ab / mean / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": (f"whole {wl.name} workload, {len(times)} passes ({sum(times):.1f} s), "
                       f"single-threaded C oracle, fp64 blend"),
            "s_per_step": mean}


# ----------------------------------------------------------------------------- GPU arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import blend_tdp_tile_gb300 as tdp

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = wk.by_name(args.workload)
    X, P, K = wk.make_inputs(wl)
    plan = tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)
    N = K.shape[2]
    s = torch.cuda.Stream(device=dev)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    with torch.cuda.stream(s):
        Xd, Pd, Kd = to_dev(X), to_dev(P), to_dev(K)
        Y, Q, mn, mx = tdp.alloc_split_outputs(plan, dev)
        keep, idx, count, kcount, Kout = tdp.alloc_filter_outputs(plan, N, dev)
        Z = torch.empty_like(Xd)
        tdp.tdp_pos_bounds(plan, Pd, mn, mx, stream=s)
        tdp.tdp_split(plan, Xd, Pd, mn, 1, Y, Q, stream=s)
        gen = torch.Generator(device=dev).manual_seed(wl.seed + 7)
        Yout = (Y.float() + wl.sigma * torch.randn(Y.shape, generator=gen, device=dev)).to(torch.bfloat16)
    s.synchronize()

    fused = args.path == "fused"

    def pre_model(Xs, Ps, Ks):
        """The pre-model stage (bounds, split, normalisation, filter) on stream s."""
        if fused:
            tdp.tdp_split_filter(plan, Xs, Ps, Ks, N, 1, Y, Q, mn, mx, keep, idx, count, kcount, Kout, stream=s)
        else:
            tdp.tdp_pos_bounds(plan, Ps, mn, mx, stream=s)
            tdp.tdp_split(plan, Xs, Ps, mn, 1, Y, Q, stream=s)
            tdp.tdp_norm_filter(plan, Ks, N, mn, mx, 1, keep, idx, count, kcount, Kout, stream=s)

    def step(evs=None):
        if evs is not None:
            evs[0].record(s)
        if fused:
            tdp.tdp_split_filter(plan, Xd, Pd, Kd, N, 1, Y, Q, mn, mx, keep, idx, count, kcount, Kout, stream=s)
        else:
            tdp.tdp_pos_bounds(plan, Pd, mn, mx, stream=s)
            if evs is not None:
                evs[3].record(s)
            tdp.tdp_split(plan, Xd, Pd, mn, 1, Y, Q, stream=s)
            if evs is not None:
                evs[4].record(s)
            tdp.tdp_norm_filter(plan, Kd, N, mn, mx, 1, keep, idx, count, kcount, Kout, stream=s)
        if evs is not None:
            evs[1].record(s)
        tdp.tdp_blend(plan, Yout, Z, stream=s)
        if evs is not None:
            evs[2].record(s)

    for _ in range(args.warmup):
        step()
    s.synchronize()
    kept_total = int(count.sum().item())
    ab = algorithmic_bytes(wl, plan.total_tile_tokens, plan.n_tiles, kept_total)

    # ---- timed region: exactly K steps, barrier + synchronize on both sides
    # Per-call CUDA events on every INSTRUMENT_EVERY-th step only: an event recorded
    # between two calls ends the programmatic-launch overlap of their kernels, so the
    # other steps run as a user's would.
    per = {i: [torch.cuda.Event(enable_timing=True) for _ in range(5)]
           for i in range(0, args.steps, INSTRUMENT_EVERY)}
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for_smi(torch, local_rank)) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(s)
    for i in range(args.steps):
        step(per.get(i))
    stop.record(s)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    if sampler:
        sampler.stop()
    ms = start.elapsed_time(stop) / args.steps
    if world > 1:
        ms = max_over_ranks(ms, dev)
    if fused:
        k_ms = {"split_filter": statistics.mean(e[0].elapsed_time(e[1]) for e in per.values())}
    else:
        k_ms = {
            "pos_bounds": statistics.mean(e[0].elapsed_time(e[3]) for e in per.values()),
            "split": statistics.mean(e[3].elapsed_time(e[4]) for e in per.values()),
            "norm_filter": statistics.mean(e[4].elapsed_time(e[1]) for e in per.values()),
        }
    k_ms["blend"] = statistics.mean(e[1].elapsed_time(e[2]) for e in per.values())

    # ---- the same step captured once in a CUDA graph and replayed (launch overhead
    # of the four calls paid once); reported beside the headline, not instead of it
    graph = None
    if rank == 0 and not args.no_graph:
        with torch.cuda.stream(s):
            step()
        s.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=s):
            step()
        for _ in range(3):
            cg.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(10, min(args.steps, 500))
        g0.record(s)
        with torch.cuda.stream(s):
            for _ in range(reps):
                cg.replay()
        g1.record(s)
        torch.cuda.synchronize()
        g_ms = g0.elapsed_time(g1) / reps
        graph = {"ms_per_step": g_ms, "value": ab["step"] / (g_ms * 1e-3) / 1e9, "unit": "GB/s", "replays": reps}
        del cg

    # ---- the other reductions over tiles (outside the headline step): conditioning
    # outputs averaged over the tiles that kept each token, audio mean over tiles
    extras = None
    if rank == 0 and not args.no_extras:
        keep2, idx2, count2, kcount2, Kout2, slot2 = tdp.alloc_filter_outputs(plan, N, dev, slot=True)
        tdp.tdp_norm_filter(plan, Kd, N, mn, mx, 1, keep2, idx2, count2, kcount2, Kout2, slot2, stream=s)
        s.synchronize()
        ncap = max(1, int(count2.max().item()))
        kept_rows = int(count2.sum().item())
        with torch.cuda.stream(s):
            Yc = torch.randn((plan.n_tiles, wl.B, ncap, wl.C), generator=gen, device=dev).to(torch.bfloat16)
            Oc = torch.empty((wl.B, N, wl.C), dtype=torch.bfloat16, device=dev)
            La = AUDIO_TOKENS * wl.C
            Au = torch.randn((plan.n_tiles, wl.B, La), generator=gen, device=dev).to(torch.bfloat16)
            Ou = torch.empty((wl.B, La), dtype=torch.bfloat16, device=dev)
        s.synchronize()
        extras = {}
        # these inputs (~70 MB) fit in L2: each timed launch follows a read of 256 MB
        # (which leaves no dirty lines), so it starts with its inputs in HBM
        flush = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
        reps = 50

        def after_flush_ms(fn):
            for _ in range(5):
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            with torch.cuda.stream(s):
                # keep the GPU busy while the host queues every launch, so that no
                # host-side gap falls between an event and its kernel
                torch.cuda._sleep(int(3e7))
                for a0, a1 in ev:
                    flush.sum()
                    a0.record(s)
                    fn()
                    a1.record(s)
            s.synchronize()
            return statistics.mean(a0.elapsed_time(a1) for a0, a1 in ev)

        for name, fn, nbytes in (
            ("cond_blend", lambda: tdp.tdp_cond_blend(plan, N, ncap, Yc, slot2, Oc, stream=s),
             kept_rows * wl.C * wl.esize + plan.n_tiles * wl.B * N * 4 + wl.B * N * wl.C * wl.esize),
            ("tile_mean", lambda: tdp.tdp_tile_mean(plan, La, Au, Ou, stream=s),
             (plan.n_tiles + 1) * wl.B * La * wl.esize)):
            t_ms = after_flush_ms(fn)
            extras[name] = {"ms": t_ms, "algorithmic_bytes": nbytes, "GB/s": nbytes / (t_ms * 1e-3) / 1e9,
                            "frac": nbytes / (t_ms * 1e-3) / 1e9 / hbm_peak()[0],
                            "timing": f"mean of {reps} launches, each after an L2 flush (256 MB read)"}
        # what the same timing gives a kernel that does almost nothing: the part of each
        # figure above that is launch and ramp, not bytes
        tiny = torch.zeros(8, device=dev)
        extras["launch_floor_ms"] = after_flush_ms(lambda: tiny.add_(1))
        extras["cond_blend"]["shape"] = f"{plan.n_tiles} tiles x {ncap} rows x {wl.C} ch, {kept_rows} kept rows"
        extras["tile_mean"]["shape"] = f"{plan.n_tiles} tiles x {AUDIO_TOKENS} audio tokens x {wl.C} ch (synthetic)"

    # ---- end to end, through the C ABI: every step copies its inputs (latent,
    # positions, cond tokens) from pinned host memory and reads its blended latent
    # back.  Three streams: step i+1's host->device copies and step i-1's
    # device->host copy overlap step i's kernels (double-buffered device inputs
    # and outputs, ordered by events).
    e2e = None
    if not args.no_e2e:
        Xh = torch.from_numpy(X.view(np.int16)).pin_memory()
        Ph = torch.from_numpy(P).pin_memory()
        Kh = torch.from_numpy(K).pin_memory()
        Zh = [torch.empty(Xd.shape, dtype=torch.int16).pin_memory() for _ in range(2)]
        Xb = [Xd, torch.empty_like(Xd)]
        Pb = [Pd, torch.empty_like(Pd)]
        Kb = [Kd, torch.empty_like(Kd)]
        Zb = [Z, torch.empty_like(Z)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_ready = [ev(), ev()]
        in_free = [ev(), ev()]
        out_ready = [ev(), ev()]
        out_free = [ev(), ev()]
        for e_ in in_free + out_free:
            e_.record(s)

        def e2e_step(i):
            j = i % 2
            with torch.cuda.stream(s_in):
                s_in.wait_event(in_free[j])
                Xb[j].view(torch.int16).copy_(Xh, non_blocking=True)
                Pb[j].copy_(Ph, non_blocking=True)
                Kb[j].copy_(Kh, non_blocking=True)
                in_ready[j].record(s_in)
            s.wait_event(in_ready[j])
            s.wait_event(out_free[j])
            pre_model(Xb[j], Pb[j], Kb[j])
            in_free[j].record(s)
            tdp.tdp_blend(plan, Yout, Zb[j], stream=s)
            out_ready[j].record(s)
            with torch.cuda.stream(s_out):
                s_out.wait_event(out_ready[j])
                Zh[j].copy_(Zb[j].view(torch.int16), non_blocking=True)
                out_free[j].record(s_out)

        for i in range(8):        # first passes over freshly pinned pages run slow
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(args.e2e_steps):
            e2e_step(i)
        s_in.wait_stream(s_out)
        e1.record(s_in)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
        # the same copies without the kernels, on the same two streams: the host
        # link's floor for this leg on this machine (reported, not subtracted)
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(s_in)
        s_out.wait_event(f0)
        for i in range(args.e2e_steps):
            j = i % 2
            with torch.cuda.stream(s_in):
                Xb[j].view(torch.int16).copy_(Xh, non_blocking=True)
                Pb[j].copy_(Ph, non_blocking=True)
                Kb[j].copy_(Kh, non_blocking=True)
            with torch.cuda.stream(s_out):
                Zh[j].copy_(Zb[j].view(torch.int16), non_blocking=True)
        s_in.wait_stream(s_out)
        f1.record(s_in)
        torch.cuda.synchronize()
        floor_ms = f0.elapsed_time(f1) / args.e2e_steps
        if world > 1:
            e2e_ms = max_over_ranks(e2e_ms, dev)
        h2d, d2h = X.nbytes + P.nbytes + K.nbytes, X.nbytes
        e2e = {"value": world * ab["step"] / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "steps": args.e2e_steps,
               "copy_floor_ms_per_step": floor_ms, "copy_floor_GBps": (h2d + d2h) / (floor_ms * 1e-3) / 1e9,
               "pipelining": "copies of steps i+1 (in) and i-1 (out) overlap step i on separate streams"}

    if rank != 0:
        return None
    peak, peak_kind = hbm_peak()
    kern = {}
    call_bytes = {"pos_bounds": ab["bounds"], "split": ab["split"], "norm_filter": ab["filter"],
                  "split_filter": ab["bounds"] + ab["split"] + ab["filter"], "blend": ab["blend"]}
    call_name = {"split_filter": "tdp_split_filter", "split": "tdp_split", "blend": "tdp_blend"}
    for name, t_ms in k_ms.items():
        b = call_bytes[name]
        gbs = b / (t_ms * 1e-3) / 1e9
        kern[name] = {"ms": t_ms, "algorithmic_bytes": b, "GB/s": gbs, "frac": gbs / peak}
    big = "split_filter" if fused else "split"
    dom = "blend" if k_ms["blend"] >= k_ms[big] else big
    call = call_name[dom]
    roof = {"bound": "hbm", "kernel": call if call != "tdp_split_filter" else
            "tdp_split_filter (tdp_bounds_init_kernel + tdp_bounds_kernel + tdp_split_filter_kernel)",
            "kernels": CALL_KERNELS[call], "achieved": kern[dom]["GB/s"], "peak": peak,
            "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s", "frac": kern[dom]["GB/s"] / peak,
            "traffic": profiled_traffic(call, wl.name), "algorithmic_bytes_per_launch": kern[dom]["algorithmic_bytes"],
            "frac_of_nominal_8tbs": kern[dom]["GB/s"] / NOMINAL_HBM_GBS}
    value = world * ab["step"] / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "dtype_detail": "bf16 latent storage, fp32 blend accumulation, int32 positions",
        "data": "synthetic", "config": config_of(wl, plan.total_tile_tokens, plan.n_tiles,
                                                 f"replicas x{world}" if world > 1 else "single GPU"),
        "frac_of_peak": value / world / peak, "frac_of_nominal_8tbs": value / world / NOMINAL_HBM_GBS,
        "latent_tokens_per_s": world * wl.B * wl.tokens / (ms * 1e-3),
        "step_algorithmic_bytes": ab["step"], "kernels": kern,
        "kernels_timing": f"CUDA events around each call on every {INSTRUMENT_EVERY}th timed step",
        "roofline": roof,
        "gpu_launches": LAUNCHES_PER_STEP[args.path] * args.steps, "path": args.path,
        "clocks": sampler.summary(t0, t1) if sampler else None,
        "e2e": e2e,
        "extra_kernels": extras,
        "graph_step": graph,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, X, P, K)
    return line


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle, as it stands, on this host: K timed steps after W warm-ups, each step
    a bounded sample of the large workload (its first Fs frames, same spatial tiling)."""
    import oracle
    oracle.build()
    wl_full = wk.by_name(args.workload)
    budget = 150.0 / max(1, args.steps + args.warmup)        # seconds per step
    probe = wl_full.replace(F=8)
    Xp, Pp, Kp = wk.make_inputs(probe)
    t8, _ = oracle_step_time(probe, Xp, Pp, Kp)
    Fs = int(min(wl_full.F, max(8, 8 * int(budget / max(t8, 1e-6)))))
    wl = wl_full.replace(F=Fs) if Fs < wl_full.F else wl_full
    X, P, K = wk.make_inputs(wl)
    box, off = oracle.plan(oracle.problem_of(wl))
    box_full, off_full = oracle.plan(oracle.problem_of(wl_full))
    times, kept = [], 0
    for _ in range(args.warmup):
        oracle_step_time(wl, X, P, K)
    for _ in range(args.steps):
        dt, kept = oracle_step_time(wl, X, P, K)
        times.append(dt)
    ab = algorithmic_bytes(wl, int(off[-1]), box.shape[0], kept)["step"]
    ms = 1e3 * sum(times) / len(times)
    value = ab / (ms * 1e-3) / 1e9
    sample = (f"{wl.name} workload cut to its first {wl.F} of {wl_full.F} frames (same H/W tiling, "
              f"2 frame tiles) per step" if wl.F < wl_full.F else f"whole {wl.name} workload per step")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl_full, int(off_full[-1]), box_full.shape[0], "host CPU, 1 thread", device=False),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=[w.name for w in wk.WORKLOADS])
    ap.add_argument("--e2e-steps", type=int, default=60)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the timing of the extra reductions")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--path", choices=["fused", "separate"], default="fused",
                    help="pre-model stage as one tdp_split_filter call, or as three calls")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
