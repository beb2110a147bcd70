"""GPU parity of the round-robin pieces of the blend ("Tiled Data Parallelism (TDP)", "What it
is": tiles are assigned to ranks round-robin and one all_reduce sums the blended tiles).

On one GPU every rank's share is computed in turn: tdp_blend_partial for rank r of `world`
against the CPU oracle's blend of that rank's tiles alone (fp32 output), the partials summed
(in the test, standing in for the collective) and stored with tdp_blend_store against the
oracle's blend of all tiles, and world == 1 against tdp_blend bit for bit."""
import numpy as np
import pytest

import oracle
import workloads as wk
from gpu_path import assert_blend_close, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


def _case(tdp, wl):
    plan = tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)
    p = oracle.problem_of(wl)
    X, P, _ = wk.make_inputs(wl)
    Y, _ = oracle.split(p, X, P)
    noise = wk.make_noise(Y.shape, wl.sigma, np.random.default_rng(wl.seed + 11))
    Yout = ((Y + noise).astype(np.float32) if wl.dtype == "f32"
            else wk.f32_to_bf16_bits(wk.bf16_bits_to_f32(Y) + noise))
    return plan, p, Yout


def _own(plan, Yout, tiles):
    own = np.zeros_like(Yout)
    for t in tiles:
        a, b = plan.B * plan.offsets[t], plan.B * plan.offsets[t + 1]
        own[a:b] = Yout[a:b]
    return own


@pytest.mark.parametrize("name,world", [("tiny", 2), ("small", 3), ("medium", 4), ("temporal", 2),
                                        ("temporal", 5), ("large", 4)])
def test_partials_sum_to_the_blend(tdp, name, world):
    import torch
    wl = wk.by_name(name)
    plan, p, Yout = _case(tdp, wl)
    Yd = to_dev(Yout)
    total = torch.zeros((wl.B, wl.F, wl.H, wl.W, wl.C), dtype=torch.float32, device="cuda")
    fp32 = wl.replace(dtype="f32")
    for r in range(world):
        Zp = torch.full_like(total, float("nan"))
        tdp.tdp_blend_partial(plan, r, world, Yd, Zp)
        torch.cuda.synchronize()
        tiles = tdp.tdp_rank_tiles(plan, r, world)
        assert list(tiles) == list(range(r, plan.n_tiles, world))
        if name != "large" or r == 0:          # one rank's partial in full on the large workload
            assert_blend_close(Zp.cpu().numpy(), oracle.blend(p, _own(plan, Yout, tiles)), fp32)
        total += Zp                            # stands in for the ranks' collective sum
    Z = torch.empty(total.shape, dtype=torch.float32 if wl.dtype == "f32" else torch.bfloat16, device="cuda")
    tdp.tdp_blend_store(plan, total, Z)
    torch.cuda.synchronize()
    assert_blend_close(to_host(Z), oracle.blend(p, Yout), wl)


@pytest.mark.parametrize("name", ["tiny", "small", "temporal"])
def test_one_rank_is_the_blend_bit_for_bit(tdp, name):
    import torch
    wl = wk.by_name(name)
    plan, p, Yout = _case(tdp, wl)
    Yd = to_dev(Yout)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    Zp = torch.empty((wl.B, wl.F, wl.H, wl.W, wl.C), dtype=torch.float32, device="cuda")
    tdp.tdp_blend_partial(plan, 0, 1, Yd, Zp)
    Z1 = torch.empty(Zp.shape, dtype=dt, device="cuda")
    tdp.tdp_blend_store(plan, Zp, Z1)
    Z2 = torch.empty_like(Z1)
    tdp.tdp_blend(plan, Yd, Z2)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(Z1), to_host(Z2))


def test_store_of_a_row_slab_and_refusals(tdp):
    import torch
    wl = wk.by_name("small")
    plan, _, _ = _case(tdp, wl)
    rows = 7
    n = rows * wl.W * wl.C
    src = torch.randn(n, dtype=torch.float32, device="cuda", generator=torch.Generator("cuda").manual_seed(1))
    dst = torch.full((n + 64,), float("nan"), dtype=torch.bfloat16, device="cuda")
    tdp.tdp_blend_store(plan, src, dst[:n])
    torch.cuda.synchronize()
    assert torch.equal(dst[:n].view(torch.int16), src.to(torch.bfloat16).view(torch.int16))
    assert torch.isnan(dst[n:].float()).all()
    Zp = torch.empty((wl.B, wl.F, wl.H, wl.W, wl.C), dtype=torch.float32, device="cuda")
    Yd = torch.zeros((wl.B * plan.total_tile_tokens, wl.C), dtype=torch.bfloat16, device="cuda")
    for rank, world in ((0, 0), (2, 2), (-1, 3)):
        with pytest.raises(tdp.TdpError, match="TDP_ERR_INVALID_ARG"):
            tdp.tdp_blend_partial(plan, rank, world, Yd, Zp)


@pytest.mark.parametrize("mode", ["reduce_scatter", "all_reduce"])
def test_blend_across_ranks_through_nccl_one_rank(tdp, mode):
    """blend_tdp_tile_gb300.ranks.blend_across_ranks end to end on the GPU: the partial blend,
    an NCCL collective over a one-rank group and the store.  With one rank every step is
    exact, so the result equals tdp_blend bit for bit."""
    import socket

    import torch
    import torch.distributed as dist

    from blend_tdp_tile_gb300 import ranks
    wl = wk.by_name("temporal")
    plan, _, Yout = _case(tdp, wl)
    Yd = to_dev(Yout)
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    group = dist.new_group(backend="nccl") if dist.is_initialized() else None
    own_init = group is None
    if own_init:
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                                device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        Z = torch.empty((wl.B, wl.F, wl.H, wl.W, wl.C), dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.Stream()
        used = ranks.blend_across_ranks(plan, Yd, Z, group=group, mode=mode, stream=s)
        s.synchronize()
        assert used == mode
        Zref = torch.empty_like(Z)
        tdp.tdp_blend(plan, Yd, Zref)
        torch.cuda.synchronize()
        assert torch.equal(Z.view(torch.int16), Zref.view(torch.int16))
    finally:
        if own_init:
            dist.destroy_process_group()
