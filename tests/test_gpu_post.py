"""tdp_blend_cond, the post-model stage in one launch ("Tiled Data Parallelism (TDP)", "What
it is" and "Shared negative (reference) positions"): its latent and conditioning-token
outputs are bit for bit those of tdp_blend and tdp_cond_blend, which the other GPU tests
compare with the CPU oracle; one case here is compared with the oracle directly."""
import numpy as np
import pytest

import oracle
import workloads as wk
from gpu_path import assert_blend_close, fill_sentinel, run_split_filter, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


def _storage(wl, shape, seed):
    x = np.random.default_rng(seed).standard_normal(shape, dtype=np.float32)
    return x if wl.dtype == "f32" else wk.f32_to_bf16_bits(x)


def _case(tdp, wl, ncap=None, seed=5):
    import torch
    X, P, K = wk.make_inputs(wl)
    plan = tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)
    out = run_split_filter(tdp, plan, wl, X, P, K, fused=True)
    N = K.shape[2]
    ncap = max(1, int(out["count"].max())) if ncap is None else ncap
    Yout = to_dev(_storage(wl, (wl.B * plan.total_tile_tokens, wl.C), seed))
    Yc = to_dev(_storage(wl, (plan.n_tiles, wl.B, ncap, wl.C), seed + 1))
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    outs = [fill_sentinel(torch.empty(shape, dtype=dt, device="cuda"))
            for shape in ((wl.B, wl.F, wl.H, wl.W, wl.C), (wl.B, N, wl.C)) * 2]
    Z1, O1, Z2, O2 = outs
    tdp.tdp_blend(plan, Yout, Z1)
    tdp.tdp_cond_blend(plan, N, ncap, Yc, out["slotd"], O1)
    tdp.tdp_blend_cond(plan, Yout, Z2, N, ncap, Yc, out["slotd"], O2)
    torch.cuda.synchronize()
    return plan, out, Yout, Yc, ncap, Z1, O1, Z2, O2


def _same(a, b):
    import torch
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("name", ["tiny", "small", "medium", "temporal", "large"])
def test_fused_post_model_matches_the_two_calls(tdp, name):
    plan, out, Yout, Yc, ncap, Z1, O1, Z2, O2 = _case(tdp, wk.by_name(name))
    assert _same(Z1, Z2), "latent differs from tdp_blend"
    assert _same(O1, O2), "conditioning outputs differ from tdp_cond_blend"


def test_fused_post_model_against_the_oracle(tdp):
    wl = wk.by_name("small")
    plan, out, Yout, Yc, ncap, Z1, O1, Z2, O2 = _case(tdp, wl)
    p = oracle.problem_of(wl)
    assert_blend_close(to_host(Z2), oracle.blend(p, to_host(Yout)), wl)
    assert_blend_close(to_host(O2), oracle.cond_blend(p, to_host(Yc), out["keep"], out["idx"], out["count"], ncap), wl)


def test_fused_post_model_truncated_rows_and_no_tokens(tdp):
    import torch
    wl = wk.by_name("temporal")
    plan, out, Yout, Yc, ncap, Z1, O1, Z2, O2 = _case(tdp, wl, ncap=7)
    assert _same(Z1, Z2) and _same(O1, O2)
    # N = 0: the blend alone
    Z3 = fill_sentinel(torch.empty_like(Z1))
    tdp.tdp_blend_cond(plan, Yout, Z3, 0, 1, None, None, None)
    torch.cuda.synchronize()
    assert _same(Z1, Z3)


def test_fused_post_model_one_row_per_tile(tdp):
    """ncap = 1: most token blocks hold no stored row and write only zeros."""
    plan, out, Yout, Yc, ncap, Z1, O1, Z2, O2 = _case(tdp, wk.by_name("medium"), ncap=1)
    assert _same(Z1, Z2) and _same(O1, O2)


def test_fused_post_model_past_the_token_block_range(tdp):
    """2048 tiles: beyond the token-block routine, the call issues the two calls in turn."""
    wl = wk.by_name("tiny").replace(F=4, H=64, W=64, C=8, dtype="bf16", num_tiles=(2, 32, 32),
                                    overlap=(1, 2, 1), n_cond=300)
    plan, out, Yout, Yc, ncap, Z1, O1, Z2, O2 = _case(tdp, wl)
    assert plan.n_tiles > 256
    assert _same(Z1, Z2) and _same(O1, O2)
