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
    "tma": 6,         # bounds init, bounds, bulk-tensor split (latent and positions), keep, compact, blend
}
# --parallel round_robin replaces the blend by tdp_blend_partial + tdp_blend_store (one more)
# ncu DRAM-traffic summaries, one per workload: profiles/dram_traffic_<workload>.txt
PROFILE_DIR = os.path.join(ROOT, "profiles")


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
    "tdp_blend_kernel": ["tdp_blend.cu", "tdp_blend_row.cuh"] + _COMMON,
    "tdp_split_kernel": ["tdp_split.cu", "tdp_filter.cuh"] + _COMMON,
    "tdp_split_filter_kernel": ["tdp_split.cu", "tdp_filter.cuh"] + _COMMON,
    "tdp_split_tma_kernel": ["tdp_split_tma.cu"] + _COMMON,
    "tdp_bounds_init_kernel": ["tdp_bounds.cu"] + _COMMON,
    "tdp_bounds_kernel": ["tdp_bounds.cu"] + _COMMON,
}
# the kernels each timed call launches
CALL_KERNELS = {
    "tdp_split_filter": ["tdp_bounds_init_kernel", "tdp_bounds_kernel", "tdp_split_filter_kernel"],
    "tdp_split": ["tdp_split_kernel"],
    "tdp_split_tma": ["tdp_split_tma_kernel"],
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


def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _oracle_worker(conn, wl):
    """One oracle process: draws the workload's inputs once, then runs one oracle pass per
    request and answers with (seconds, kept tokens)."""
    X, P, K = wk.make_inputs(wl)
    conn.send("ready")
    while True:
        msg = conn.recv()
        if msg is None:
            break
        conn.send(oracle_step_time(wl, X, P, K))
    conn.close()


class OraclePool:
    """`n` processes (spawn start method: the parent may already hold a CUDA context), each
    running the oracle as it stands, single-threaded, on its own copy of workload `wl`.  A
    step sends every process one pass at once and ends when the last one is done, so
    n passes over the workload take the slowest process's time."""

    def __init__(self, wl, n):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.n, self.wl = n, wl
        self.conns, self.procs = [], []
        for _ in range(n):
            a, b = ctx.Pipe()
            pr = ctx.Process(target=_oracle_worker, args=(b, wl), daemon=True)
            pr.start()
            self.conns.append(a)
            self.procs.append(pr)
        for c in self.conns:
            assert c.recv() == "ready"

    def step(self):
        """(wall seconds of one pass on every process, kept tokens of one pass)."""
        t = time.perf_counter()
        for c in self.conns:
            c.send("pass")
        res = [c.recv() for c in self.conns]
        return time.perf_counter() - t, res[0][1]

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except OSError:
                pass
        for pr in self.procs:
            pr.join(timeout=30)
            if pr.is_alive():
                pr.kill()


def oracle_pool(wl_full, seconds_per_step, n):
    """(OraclePool of `n` processes, the workload each runs): the workload cut to its first
    frames (same H/W tiling) so that one round -- one pass in every process at once --
    takes about `seconds_per_step`, sized from a round on an 8-frame probe (the processes
    share the host's memory bandwidth, so a round is slower than one pass alone)."""
    import oracle
    probe = wl_full.replace(F=min(8, wl_full.F))
    pool = OraclePool(probe, n)
    try:
        pool.step()
        t8 = pool.step()[0]
    finally:
        pool.close()
    Fs = int(min(wl_full.F, max(probe.F, probe.F * int(seconds_per_step / max(t8, 1e-6)))))
    wl = wl_full
    if Fs < wl_full.F:
        try:
            oracle.plan(oracle.problem_of(wl_full.replace(F=Fs)))     # the tiling must stay valid
            wl = wl_full.replace(F=Fs)
        except ValueError:
            pass
    return OraclePool(wl, n), wl


def sample_words(wl, wl_full):
    return (f"first {wl.F} of {wl_full.F} frames (same H/W tiling)" if wl.F < wl_full.F
            else "whole workload")


def cpu_baseline(wl, X, P, K, seconds=12.0):
    """The oracle timed on this host's cores: `host_cores()` processes at once, each on a
    bounded sample of the workload (its first frames), plus one core on the whole workload."""
    import oracle
    oracle.build()
    box, off = oracle.plan(oracle.problem_of(wl))
    # one core, whole workload
    times, kept = [], 0
    while (sum(times) < seconds / 2 and len(times) < 10) or len(times) < 2:
        dt, kept = oracle_step_time(wl, X, P, K)
        times.append(dt)
    ab1 = algorithmic_bytes(wl, int(off[-1]), box.shape[0], kept)["step"]
    single = {"value": ab1 / (sum(times) / len(times)) / 1e9, "unit": "GB/s", "cores": 1,
              "sample": f"whole {wl.name} workload, {len(times)} passes ({sum(times):.1f} s)"}
    # every core, one sample per process
    n = host_cores()
    pool, ws = oracle_pool(wl, 1.0, n)
    bs, offs = oracle.plan(oracle.problem_of(ws))
    try:
        pool.step()                                   # first touch of every process's pages
        steps, kept_s = [], 0
        while sum(steps) < seconds / 2 or len(steps) < 2:
            dt, kept_s = pool.step()
            steps.append(dt)
    finally:
        pool.close()
    abs_ = algorithmic_bytes(ws, int(offs[-1]), bs.shape[0], kept_s)["step"]
    mean = sum(steps) / len(steps)
    return {"value": n * abs_ / mean / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": (f"{n} single-threaded oracle processes at once, each on the {wl.name} workload "
                       f"({sample_words(ws, wl)}); {len(steps)} rounds of one pass in each process "
                       f"({sum(steps):.1f} s); fp64 blend"),
            "s_per_round": mean, "single_core": single}


# ----------------------------------------------------------------------------- GPU arm
PER_CALL_REPS = 100          # launches each per-call figure averages


class DeviceCase:
    """One workload resident on the device: inputs, every output buffer, the tile outputs
    fed to the blend (split tiles + N(0, sigma) noise, made once) and the library calls of
    the hot path bound to them, all on stream `s`."""

    def __init__(self, tdp, torch, wl, dev, s, X=None, P=None, K=None):
        self.tdp, self.torch, self.wl, self.s = tdp, torch, wl, s
        if X is None:
            X, P, K = wk.make_inputs(wl)
        self.X, self.P, self.K = X, P, K
        self.plan = tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)
        self.N = K.shape[2]
        with torch.cuda.stream(s):
            self.Xd, self.Pd, self.Kd = self.to_dev(X, dev), self.to_dev(P, dev), self.to_dev(K, dev)
            self.Y, self.Q, self.mn, self.mx = tdp.alloc_split_outputs(self.plan, dev)
            (self.keep, self.idx, self.count, self.kcount,
             self.Kout) = tdp.alloc_filter_outputs(self.plan, self.N, dev)
            self.Z = torch.empty_like(self.Xd)
            tdp.tdp_pos_bounds(self.plan, self.Pd, self.mn, self.mx, stream=s)
            tdp.tdp_split(self.plan, self.Xd, self.Pd, self.mn, 1, self.Y, self.Q, stream=s)
            gen = torch.Generator(device=dev).manual_seed(wl.seed + 7)
            self.gen = gen
            noise = wl.sigma * torch.randn(self.Y.shape, generator=gen, device=dev)
            self.Yout = (self.Y.float() + noise).to(self.Y.dtype)
            del noise
        s.synchronize()
        self.split_filter()
        s.synchronize()
        self.kept = int(self.count.sum().item())
        self.ab = algorithmic_bytes(wl, self.plan.total_tile_tokens, self.plan.n_tiles, self.kept)

    @staticmethod
    def to_dev(a, dev):
        import torch
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    # the calls of one step
    def split_filter(self, X=None, P=None, K=None):
        self.tdp.tdp_split_filter(self.plan, self.Xd if X is None else X, self.Pd if P is None else P,
                                  self.Kd if K is None else K, self.N, 1, self.Y, self.Q, self.mn, self.mx,
                                  self.keep, self.idx, self.count, self.kcount, self.Kout, stream=self.s)

    def pos_bounds(self, P=None):
        self.tdp.tdp_pos_bounds(self.plan, self.Pd if P is None else P, self.mn, self.mx, stream=self.s)

    def split(self, X=None, P=None):
        self.tdp.tdp_split(self.plan, self.Xd if X is None else X, self.Pd if P is None else P, self.mn, 1,
                           self.Y, self.Q, stream=self.s)

    def split_tma(self, X=None, P=None):
        self.tdp.tdp_split_tma(self.plan, self.Xd if X is None else X, self.Pd if P is None else P, self.mn, 1,
                               self.Y, self.Q, stream=self.s)

    def norm_filter(self, K=None):
        self.tdp.tdp_norm_filter(self.plan, self.Kd if K is None else K, self.N, self.mn, self.mx, 1, self.keep,
                                 self.idx, self.count, self.kcount, self.Kout, stream=self.s)

    blend_impl = None        # replaces tdp_blend when set (the round-robin ranks' blend)

    def blend(self, Z=None):
        if self.blend_impl is not None:
            self.blend_impl(self.Z if Z is None else Z)
        else:
            self.tdp.tdp_blend(self.plan, self.Yout, self.Z if Z is None else Z, stream=self.s)

    def pre_model(self, path, X=None, P=None, K=None):
        if path == "fused":
            self.split_filter(X, P, K)
        else:
            self.pos_bounds(P)
            (self.split_tma if path == "tma" else self.split)(X, P)
            self.norm_filter(K)

    def step(self, path):
        self.pre_model(path)
        self.blend()

    def inputs_fit_l2(self):
        return self.wl.B * self.plan.total_tile_tokens * self.wl.C * self.wl.esize <= L2_BYTES


class L2Flush:
    """Empties L2 between timed launches: a write of 256 MB (twice L2) and then a read of
    another 256 MB, so that the next launch starts with its inputs in HBM and no dirty
    lines of the flush left to write back inside its interval."""

    def __init__(self, torch, dev):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.fill_(1)
        self.r.sum()


def call_ms(torch, s, fn, reps=PER_CALL_REPS, flush=None):
    """Mean device time of one call of `fn` on stream `s` (with the median of the same launches
    as .median): `reps` launches, each bracketed by CUDA events on `s` (and, with `flush`,
    each after an L2 flush).  The GPU is kept busy while the host queues them, so host-side
    launch work never falls inside an interval."""
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    s.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(s):
        torch.cuda._sleep(int(4e7))
        for a0, a1 in ev:
            if flush is not None:
                flush()
            a0.record(s)
            fn()
            a1.record(s)
    s.synchronize()
    times = [a0.elapsed_time(a1) for a0, a1 in ev]
    return TimedMs(statistics.mean(times), statistics.median(times))


class TimedMs(float):
    """A mean time in ms (the float) that also carries the median of the same launches."""

    def __new__(cls, mean, median):
        obj = super().__new__(cls, mean)
        obj.median = median
        return obj


def rotating_ms(torch, s, fns, reps):
    """Mean device time per launch of calls issued back to back on stream `s`, launch i running
    fns[i % len(fns)]: each callable works on its own set of buffers, and the sets together
    are several times L2, so a set's inputs have left L2 before it comes round again.  One
    event pair brackets all `reps` launches (the launches overlap as they do in a loop)."""
    with torch.cuda.stream(s):
        for fn in fns:
            fn()
    s.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        torch.cuda._sleep(int(4e7))
        e0.record(s)
        for i in range(reps):
            fns[i % len(fns)]()
        e1.record(s)
    s.synchronize()
    return e0.elapsed_time(e1) / reps


def call_entry(t_ms, nbytes, peak):
    gbs = nbytes / (t_ms * 1e-3) / 1e9
    e = {"ms": float(t_ms), "algorithmic_bytes": nbytes, "GB/s": gbs, "frac": gbs / peak,
         "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS}
    if isinstance(t_ms, TimedMs):
        e["ms_median"] = t_ms.median
    return e


def time_calls(case, torch, peak, flush=None, reps=PER_CALL_REPS):
    """Per-call device times of every call of the hot path on one workload."""
    ab, s = case.ab, case.s
    out = {
        "split_filter": call_entry(call_ms(torch, s, case.split_filter, reps, flush),
                                   ab["bounds"] + ab["split"] + ab["filter"], peak),
        "pos_bounds": call_entry(call_ms(torch, s, case.pos_bounds, reps, flush), ab["bounds"], peak),
        "split": call_entry(call_ms(torch, s, case.split, reps, flush), ab["split"], peak),
        "split_tma": call_entry(call_ms(torch, s, case.split_tma, reps, flush), ab["split"], peak),
        "norm_filter": call_entry(call_ms(torch, s, case.norm_filter, reps, flush), ab["filter"], peak),
        "blend": call_entry(call_ms(torch, s, case.blend, reps, flush), ab["blend"], peak),
    }
    out["step"] = call_entry(call_ms(torch, s, lambda: case.step("fused"), reps, flush), ab["step"], peak)
    out["step"]["latent_tokens_per_s"] = case.wl.B * case.wl.tokens / (out["step"]["ms"] * 1e-3)
    return out


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
    s = torch.cuda.Stream(device=dev)
    case = DeviceCase(tdp, torch, wl, dev, s, X, P, K)
    plan, N, gen = case.plan, case.N, case.gen
    Xd, Pd, Kd, Z, Yout = case.Xd, case.Pd, case.Kd, case.Z, case.Yout
    mn, mx = case.mn, case.mx
    path = args.path
    peak, peak_kind = hbm_peak()
    rr = args.parallel == "round_robin"
    if rr:
        # every rank splits the whole latent and holds every tile's output (the stand-in
        # model); the blend reads only this rank's tiles and the collective sums the ranks
        from blend_tdp_tile_gb300 import ranks
        Zp = torch.empty(Z.shape, dtype=torch.float32, device=dev)
        case.blend_impl = lambda Zout: ranks.blend_across_ranks(plan, Yout, Zout, mode=args.collective, Zp=Zp,
                                                                stream=s)

    def step():
        case.step(path)

    def pre_model(Xs, Ps, Ks):
        """The pre-model stage (bounds, split, normalisation, filter) on stream s."""
        case.pre_model(path, Xs, Ps, Ks)

    for _ in range(args.warmup):
        step()
    s.synchronize()
    ab = case.ab

    # ---- timed region: exactly K steps, barrier + synchronize on both sides, no event
    # between the calls (an event would end the programmatic-launch overlap of the kernels)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for_smi(torch, local_rank)) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(s)
    for _ in range(args.steps):
        step()
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

    # ---- every call of the hot path timed on its own, after the timed region
    kern = time_calls(case, torch, peak) if rank == 0 or rr else {}

    # ---- the same step captured once in a CUDA graph and replayed (launch overhead
    # of the four calls paid once); reported beside the headline, not instead of it
    graph = None
    if rank == 0 and not args.no_graph and not rr:
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
        # these inputs (~70 MB) fit in L2: each timed launch follows an L2 flush
        flush = L2Flush(torch, dev)
        reps = 50
        for name, fn, nbytes in (
            ("cond_blend", lambda: tdp.tdp_cond_blend(plan, N, ncap, Yc, slot2, Oc, stream=s),
             kept_rows * wl.C * wl.esize + plan.n_tiles * wl.B * N * 4 + wl.B * N * wl.C * wl.esize),
            ("tile_mean", lambda: tdp.tdp_tile_mean(plan, La, Au, Ou, stream=s),
             (plan.n_tiles + 1) * wl.B * La * wl.esize)):
            extras[name] = call_entry(call_ms(torch, s, fn, reps, flush), nbytes, peak)
            extras[name]["timing"] = f"mean of {reps} launches, each after an L2 flush"
        # the post-model stage in one call (blend + conditioning blend, one launch) against
        # the same two calls one after the other
        cond_bytes = extras["cond_blend"]["algorithmic_bytes"]
        Zx = torch.empty_like(Z)
        fused_ms = call_ms(torch, s, lambda: tdp.tdp_blend_cond(plan, Yout, Zx, N, ncap, Yc, slot2, Oc, stream=s),
                           reps, flush)
        pair_ms = call_ms(torch, s, lambda: (tdp.tdp_blend(plan, Yout, Zx, stream=s),
                                             tdp.tdp_cond_blend(plan, N, ncap, Yc, slot2, Oc, stream=s)), reps, flush)
        extras["blend_cond"] = call_entry(fused_ms, ab["blend"] + cond_bytes, peak)
        extras["blend_cond"].update({"two_calls_ms": pair_ms,
                                     "timing": f"mean of {reps} launches, each after an L2 flush",
                                     "calls": "tdp_blend_cond (one launch) against tdp_blend + tdp_cond_blend"})
        del Zx
        # what the same timing gives a kernel that does almost nothing: the part of each
        # figure above that is launch and ramp, not bytes
        tiny = torch.zeros(8, device=dev)
        extras["launch_floor_ms"] = call_ms(torch, s, lambda: tiny.add_(1), reps, flush)
        del flush
        extras["cond_blend"]["shape"] = f"{plan.n_tiles} tiles x {ncap} rows x {wl.C} ch, {kept_rows} kept rows"
        # the same reduction in two calls: the records made once (the conditioning tokens do
        # not change between denoising steps), then each step's call from the records
        if plan.n_tiles <= 256:
            recs = torch.empty(tdp.tdp_cond_records_size(plan, N), dtype=torch.int32, device=dev)
            flush = L2Flush(torch, dev)
            rec_ms = call_ms(torch, s, lambda: tdp.tdp_cond_records(plan, N, ncap, slot2, recs, stream=s), 10, flush)
            nblk = wl.B * ((N + 7) // 8)
            rec_bytes = (kept_rows * wl.C * wl.esize + nblk * 26 * 4 + kept_rows * 4 + wl.B * N * wl.C * wl.esize)
            extras["cond_blend_records"] = call_entry(
                call_ms(torch, s, lambda: tdp.tdp_cond_blend_records(plan, N, recs, Yc, ncap, Oc, stream=s), reps,
                        flush), rec_bytes, peak)
            extras["cond_blend_records"].update({
                "timing": f"mean of {reps} launches, each after an L2 flush",
                "bytes": "kept rows + the records' headers and row numbers + out (the slots are not read)",
                "records_ms": rec_ms, "records": "tdp_cond_records, once per set of conditioning tokens (mean of 10)"})
            del flush, recs
        extras["tile_mean"]["shape"] = f"{plan.n_tiles} tiles x {AUDIO_TOKENS} audio tokens x {wl.C} ch (synthetic)"
        # the same calls launched back to back, as in a denoising loop, each launch on its own
        # copy of the inputs: enough copies to fill L2 three times over, so no launch finds its
        # inputs in L2 and no flush or event sits between launches
        set_bytes = max(Yc.numel() * Yc.element_size() + slot2.numel() * 4, Au.numel() * Au.element_size())
        nsets = min(16, max(4, -(-3 * L2_BYTES // set_bytes)))
        b2b_reps = 20 * nsets
        with torch.cuda.stream(s):
            Ycs = [Yc.clone() for _ in range(nsets)]
            slots = [slot2.clone() for _ in range(nsets)]
            Ocs = [torch.empty_like(Oc) for _ in range(nsets)]
            Aus = [Au.clone() for _ in range(nsets)]
            Ous = [torch.empty_like(Ou) for _ in range(nsets)]
        s.synchronize()
        b2b = {"cond_blend": [lambda i=i: tdp.tdp_cond_blend(plan, N, ncap, Ycs[i], slots[i], Ocs[i], stream=s)
                              for i in range(nsets)],
               "tile_mean": [lambda i=i: tdp.tdp_tile_mean(plan, La, Aus[i], Ous[i], stream=s) for i in range(nsets)]}
        if "cond_blend_records" in extras:
            recss = [torch.empty(tdp.tdp_cond_records_size(plan, N), dtype=torch.int32, device=dev)
                     for _ in range(nsets)]
            for i in range(nsets):
                tdp.tdp_cond_records(plan, N, ncap, slots[i], recss[i], stream=s)
            b2b["cond_blend_records"] = [
                lambda i=i: tdp.tdp_cond_blend_records(plan, N, recss[i], Ycs[i], ncap, Ocs[i], stream=s)
                for i in range(nsets)]
        for name, fns in b2b.items():
            e = call_entry(rotating_ms(torch, s, fns, b2b_reps), extras[name]["algorithmic_bytes"], peak)
            e["timing"] = (f"{b2b_reps} launches back to back between one event pair, launch i on input set "
                           f"i % {nsets} ({nsets} sets of {set_bytes / 1e6:.0f} MB: no launch finds its inputs in L2)")
            extras[name]["back_to_back"] = e
        del Ycs, slots, Ocs, Aus, Ous, b2b
        if "cond_blend_records" in extras:
            del recss

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
            case.blend(Zb[j])
            out_ready[j].record(s)
            with torch.cuda.stream(s_out):
                s_out.wait_event(out_ready[j])
                Zh[j].copy_(Zb[j].view(torch.int16), non_blocking=True)
                out_free[j].record(s_out)

        def copies_only(n):
            """The same copies without the kernels, on the same two streams: the host link's
            floor for this leg on this machine (reported, not subtracted)."""
            torch.cuda.synchronize()
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(s_in)
            s_out.wait_event(f0)
            for i in range(n):
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
            return f0.elapsed_time(f1) / n

        # first passes over freshly pinned pages run slow: the copies alone, then steps
        copies_only(8)
        for i in range(16):
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
        floor_ms = copies_only(args.e2e_steps)
        if world > 1:
            e2e_ms = max_over_ranks(e2e_ms, dev)
        h2d, d2h = X.nbytes + P.nbytes + K.nbytes, X.nbytes
        e2e = {"value": (1 if rr else world) * ab["step"] / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "steps": args.e2e_steps,
               "copy_floor_ms_per_step": floor_ms, "copy_floor_GBps": (h2d + d2h) / (floor_ms * 1e-3) / 1e9,
               "pipelining": "copies of steps i+1 (in) and i-1 (out) overlap step i on separate streams"}

    if rank != 0:
        return None
    call_name = {"split_filter": "tdp_split_filter", "split": "tdp_split", "split_tma": "tdp_split_tma",
                 "blend": "tdp_blend"}
    big = {"fused": "split_filter", "separate": "split", "tma": "split_tma"}[path]
    dom = "blend" if kern["blend"]["ms"] >= kern[big]["ms"] else big
    call = call_name[dom]
    roof = {"bound": "hbm", "kernel": call if call != "tdp_split_filter" else
            "tdp_split_filter (tdp_bounds_init_kernel + tdp_bounds_kernel + tdp_split_filter_kernel)",
            "kernels": CALL_KERNELS[call], "achieved": kern[dom]["GB/s"], "peak": peak,
            "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s", "frac": kern[dom]["frac"],
            "traffic": profiled_traffic(call, wl.name), "algorithmic_bytes_per_launch": kern[dom]["algorithmic_bytes"],
            "frac_of_nominal_8tbs": kern[dom]["frac_of_nominal_8tbs"],
            "timing": f"mean of {PER_CALL_REPS} launches of the call (ms_median beside), CUDA events on its stream"}

    # ---- every workload: each call timed the same way; inputs that fit in L2 are
    # flushed out of it before every launch
    per_workload = None
    if not args.no_per_workload and not rr:
        per_workload = {}
        flush = L2Flush(torch, dev)
        for w in wk.WORKLOADS:
            if w.name == wl.name:
                c, fl = case, None
            else:
                c = DeviceCase(tdp, torch, w, dev, s)
                fl = flush if c.wl.B * c.wl.tokens * c.wl.C * c.wl.esize < 2 * L2_BYTES else None
            calls = kern if c is case else time_calls(c, torch, peak, flush=fl)
            per_workload[w.name] = {
                "config": config_of(w, c.plan.total_tile_tokens, c.plan.n_tiles, "single GPU")["workload"],
                "l2": "flushed before every launch" if fl is not None else "inputs larger than L2; no flush",
                "calls": {k: dict({"ms": v["ms"], "GB/s": v["GB/s"], "frac": v["frac"],
                                   "frac_of_nominal_8tbs": v["frac_of_nominal_8tbs"]},
                                  **({"ms_median": v["ms_median"]} if "ms_median" in v else {}),
                                  **({"traffic": profiled_traffic("tdp_" + k, w.name)}
                                     if "tdp_" + k in CALL_KERNELS else {}))
                          for k, v in calls.items()},
                "latent_tokens_per_s": calls["step"]["latent_tokens_per_s"],
            }
            if fl is not None:
                # the same calls without the flush: launches back to back on inputs left in L2
                warm = time_calls(c, torch, peak)
                per_workload[w.name]["calls_without_flush"] = {
                    "note": "no flush between launches: inputs resident in L2, not an HBM measurement",
                    **{k: {"ms": v["ms"], "GB/s": v["GB/s"]} for k, v in warm.items()}}
            if c is not case:
                del c
                torch.cuda.empty_cache()
        del flush
    problems = 1 if rr else world           # round-robin: one problem over all ranks
    value = problems * ab["step"] / (ms * 1e-3) / 1e9
    if rr:
        parallelism = f"round-robin tiles over {world} rank(s), {args.collective} of fp32 partials"
    else:
        parallelism = f"replicas x{world}" if world > 1 else "single GPU"
    launches = LAUNCHES_PER_STEP[args.path] + (1 if rr else 0)       # partial blend + store for the blend
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "strong" if rr else "weak",
        "vs_baseline": None, "dtype": "bf16",
        "dtype_detail": "bf16 latent storage, fp32 blend accumulation, int32 positions",
        "data": "synthetic", "config": config_of(wl, plan.total_tile_tokens, plan.n_tiles, parallelism),
        "frac_of_peak": value / world / peak, "frac_of_nominal_8tbs": value / world / NOMINAL_HBM_GBS,
        "latent_tokens_per_s": problems * wl.B * wl.tokens / (ms * 1e-3),
        "step_algorithmic_bytes": ab["step"], "kernels": kern,
        "kernels_timing": (f"after the timed region: mean of {PER_CALL_REPS} launches of each call, CUDA events "
                           f"on its stream around each launch, the GPU kept busy while the host queued them"),
        "roofline": roof,
        "gpu_launches": launches * args.steps, "path": args.path,
        "clocks": sampler.summary(t0, t1) if sampler else None,
        "e2e": e2e,
        "extra_kernels": extras,
        "graph_step": graph,
        "per_workload": per_workload,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, X, P, K)
    return line


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle, as it stands, on this host's cores: K timed steps after W warm-ups.
    A step runs one oracle pass in each of `host_cores()` single-threaded processes at once,
    each on a bounded sample of the workload (its first frames, same spatial tiling), so
    that the whole run stays within a few minutes."""
    import oracle
    oracle.build()
    wl_full = wk.by_name(args.workload)
    budget = 150.0 / max(1, args.steps + args.warmup)        # seconds per step
    n = host_cores()
    pool, wl = oracle_pool(wl_full, budget, n)
    box, off = oracle.plan(oracle.problem_of(wl))
    box_full, off_full = oracle.plan(oracle.problem_of(wl_full))
    times, kept = [], 0
    try:
        for _ in range(args.warmup):
            pool.step()
        for _ in range(args.steps):
            dt, kept = pool.step()
            times.append(dt)
    finally:
        pool.close()
    ab = n * algorithmic_bytes(wl, int(off[-1]), box.shape[0], kept)["step"]
    ms = 1e3 * sum(times) / len(times)
    value = ab / (ms * 1e-3) / 1e9
    sample = (f"{n} single-threaded oracle processes at once, each running one pass over the {wl.name} "
              f"workload ({sample_words(wl, wl_full)}) per step")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl_full, int(off_full[-1]), box_full.shape[0], f"host CPU, {n} processes",
                            device=False),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
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
    ap.add_argument("--no-per-workload", action="store_true", help="skip the per-call timing of every workload")
    ap.add_argument("--parallel", choices=["replicas", "round_robin"], default="replicas",
                    help="replicas: every rank runs the whole step on its own problem (weak scaling); "
                         "round_robin: the ranks share one problem, tile t blended on rank t %% N and the "
                         "partials summed by a collective (strong scaling)")
    ap.add_argument("--collective", choices=["reduce_scatter", "all_reduce"], default="reduce_scatter",
                    help="collective of the round_robin blend")
    ap.add_argument("--path", choices=["fused", "separate", "tma"], default="fused",
                    help="pre-model stage as one tdp_split_filter call, as three calls, or as three calls "
                         "with the bulk-tensor split (tdp_split_tma)")
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

    distributed = world > 1 or args.parallel == "round_robin"
    if distributed:
        import torch
        import torch.distributed as dist
        if "MASTER_ADDR" not in os.environ:          # one rank started without torchrun
            import socket
            with socket.socket() as sk:
                sk.bind(("127.0.0.1", 0))
                port = sk.getsockname()[1]
            os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK="0", WORLD_SIZE="1")
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    # stdout carries the one JSON line: whatever the libraries print while the arm runs
    # (NCCL's version banner, for one) goes to stderr
    sys.stdout.flush()
    saved = os.dup(1)
    os.dup2(2, 1)
    try:
        line = run_ours(args, rank, world, local_rank)
        if distributed:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
    finally:
        sys.stdout.flush()
        # C stdio buffers (NCCL writes its banner through them) are flushed here, while
        # fd 1 still points at stderr, not at exit after the JSON line
        import ctypes
        ctypes.CDLL(None).fflush(None)
        os.dup2(saved, 1)
        os.close(saved)
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
