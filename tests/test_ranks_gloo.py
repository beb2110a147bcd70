"""Multi-process logic on CPU (gloo, world size 2).

- bench.py: the timing is the maximum over ranks, and the reference arm runs on rank 0 only.
- Round-robin TDP across ranks ("Tiled Data Parallelism (TDP)", "What it is": tiles go to
  ranks round-robin and one all_reduce sums the blended tiles): each rank takes the tiles
  the library's tdp_rank_tiles gives it, blends them alone (here with the CPU oracle, which
  stands in for tdp_blend_partial, the one step that needs a GPU), and
  blend_tdp_tile_gb300.ranks.reduce_partials sums the ranks' partials with the collective
  and stores the result; every rank must end with the oracle's blend of all tiles."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(1.5 + rank * 2.0, "cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 3.5, 1: 3.5}


def test_reference_arm_other_ranks_do_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def _blend_worker(rank, world, port, q, name, mode, overrides):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch
    import torch.distributed as dist

    import blend_tdp_tile_gb300 as tdp
    import oracle
    import workloads as wk
    from blend_tdp_tile_gb300 import ranks
    from gpu_path import assert_blend_close
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _blend_rank(rank, world, q, name, mode, overrides, np, torch, tdp, oracle, wk, ranks, assert_blend_close)
    except BaseException as e:          # report instead of leaving the parent waiting
        q.put((rank, "error", repr(e), b""))
        raise
    finally:
        dist.destroy_process_group()


def _blend_rank(rank, world, q, name, mode, overrides, np, torch, tdp, oracle, wk, ranks, assert_blend_close):
    wl = wk.by_name(name).replace(**overrides)
    plan = tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)
    p = oracle.problem_of(wl)
    X, P, _ = wk.make_inputs(wl)
    Y, _ = oracle.split(p, X, P)
    noise = wk.make_noise(Y.shape, wl.sigma, np.random.default_rng(wl.seed + 5))
    Yout = ((Y + noise).astype(np.float32) if wl.dtype == "f32"
            else wk.f32_to_bf16_bits(wk.bf16_bits_to_f32(Y) + noise))
    mine = tdp.tdp_rank_tiles(plan, rank, world)
    # this rank's tile outputs only: the other tiles' rows are zero
    own = np.zeros_like(Yout)
    for t in mine:
        a, b = plan.B * plan.offsets[t], plan.B * plan.offsets[t + 1]
        own[a:b] = Yout[a:b]
    Zp = torch.from_numpy(oracle.blend(p, own).astype(np.float32))
    tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    Z = torch.empty(Zp.shape, dtype=tdt)
    used = ranks.reduce_partials(Zp, Z, wl.W * wl.C, lambda src, dst: dst.copy_(src.to(dst.dtype)), mode=mode)
    z = Z.view(torch.int16).numpy().view(np.uint16) if wl.dtype == "bf16" else Z.numpy()
    assert_blend_close(z, oracle.blend(p, Yout), wl)
    q.put((rank, used, sorted(int(t) for t in mine), z.tobytes()))


@pytest.mark.parametrize("name,mode,overrides,expect", [
    ("tiny", "all_reduce", {}, "all_reduce"),
    ("tiny", "reduce_scatter", {}, "reduce_scatter"),
    ("small", "reduce_scatter", dict(F=4, n_cond=8), "reduce_scatter"),
    ("temporal", "reduce_scatter", dict(B=1, F=9, H=27, W=30, C=16, n_cond=8), "all_reduce"),  # 243 rows: odd
])
def test_round_robin_blend_across_two_ranks(name, mode, overrides, expect):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_blend_worker, args=(r, 2, port, q, name, mode, overrides)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict((r, rest) for r, *rest in (q.get(timeout=300) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        assert got[r][0] != "error", f"rank {r}: {got[r][1]}"
    (m0, t0, z0), (m1, t1, z1) = got[0], got[1]
    assert m0 == m1 == expect
    assert not set(t0) & set(t1) and sorted(t0 + t1) == list(range(len(t0) + len(t1)))   # each tile once
    assert all(t % 2 == 0 for t in t0) and all(t % 2 == 1 for t in t1)                   # round-robin
    assert z0 == z1                                                                        # same latent on both
