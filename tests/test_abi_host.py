"""CPU-side checks of the C ABI: the library loads, exports every function the
header declares, and its host-only plan logic agrees with the oracle and
refuses invalid problems with the documented status (no GPU needed: plan
creation makes no CUDA call)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads as wk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# Tests that hand the library fake pointer values check that the host refuses them
# before any launch; they run only where no GPU is present, so that a validation bug
# can never turn into a kernel launch on a bogus address.
no_gpu_only = pytest.mark.skipif(_has_gpu(), reason="fake-pointer checks run only without a GPU")


@pytest.fixture(scope="module")
def tdp():
    import __graft_entry__
    __graft_entry__.build()
    import blend_tdp_tile_gb300
    return blend_tdp_tile_gb300


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(tdp_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("tdp_plan_create", "tdp_plan_info", "tdp_plan_destroy", "tdp_split",
                     "tdp_norm_filter", "tdp_split_filter", "tdp_blend", "tdp_status_str"):
        assert required in names


def test_library_exports_every_declared_symbol(tdp):
    lib = ctypes.CDLL(tdp.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_plan_matches_oracle(tdp, wl):
    plan = tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)
    box, off = oracle.plan(oracle.problem_of(wl))
    nt, tot, boxes, offsets = tdp.tdp_plan_info(plan)
    assert nt == box.shape[0] and tot == off[-1]
    assert np.array_equal(boxes, box) and np.array_equal(offsets, off)


def test_plan_matches_oracle_sweep(tdp):
    rng = np.random.default_rng(0)
    for _ in range(300):
        L = [int(rng.integers(1, 40)) for _ in range(3)]
        n = [int(rng.integers(1, 7)) for _ in range(3)]
        o = [int(rng.integers(0, 6)) for _ in range(3)]
        try:
            box, off = oracle.plan(oracle.problem(1, *L, 8, 4, n, o))
        except ValueError:
            with pytest.raises(tdp.TdpError) as ei:
                tdp.tdp_plan_create(1, *L, 8, "f32", n, o)
            assert ei.value.status in (2, 5)
            continue
        plan = tdp.tdp_plan_create(1, *L, 8, "f32", n, o)
        assert np.array_equal(plan.boxes, box) and np.array_equal(plan.offsets, off)


@pytest.mark.parametrize("kw,status", [
    (dict(C=6, dtype="bf16"), 4),                      # 12-byte rows: not a multiple of 16
    (dict(C=2, dtype="f32"), 4),
    (dict(num_tiles=(1, 9, 1)), 2),                    # more tiles than cells
    (dict(num_tiles=(1, 2, 2), overlap=(0, 5, 2)), 2),  # overlap longer than a core
    (dict(overlap=(0, -1, 0)), 2),
    (dict(num_tiles=(0, 1, 1)), 2),
    (dict(W=200, num_tiles=(1, 1, 65), overlap=(0, 0, 0)), 5),
    (dict(B=-1), 1),
    (dict(F=0), 1),
    (dict(F=(1 << 25) + 1, num_tiles=(1, 1, 1), overlap=(0, 0, 0)), 5),       # a dimension past 2^25
    (dict(B=1 << 16, F=256, H=256, num_tiles=(1, 1, 1), overlap=(0, 0, 0)), 5),   # B*F*H rows past 2^31
    (dict(B=1 << 13, F=64, H=64, W=64, num_tiles=(64, 64, 64), overlap=(0, 0, 0)), 5),  # nt*B*3 past 2^31
])
def test_plan_rejects_invalid(tdp, kw, status):
    base = dict(B=1, F=3, H=8, W=12, C=16, dtype="f32", num_tiles=(1, 2, 2), overlap=(0, 2, 2))
    base.update(kw)
    with pytest.raises(tdp.TdpError) as ei:
        tdp.tdp_plan_create(base["B"], base["F"], base["H"], base["W"], base["C"], base["dtype"],
                            base["num_tiles"], base["overlap"])
    assert ei.value.status == status
    assert tdp.tdp_last_error_detail()


@no_gpu_only
def test_bad_dtype_and_null_args(tdp):
    lib = ctypes.CDLL(tdp.LIB_PATH)
    pr = tdp._Problem()
    pr.B, pr.F, pr.H, pr.W, pr.C, pr.dtype = 1, 3, 8, 12, 16, 7
    for d in range(3):
        pr.dim[d].num_tiles, pr.dim[d].overlap = 1, 0
    h = ctypes.c_void_p()
    lib.tdp_plan_create.argtypes = [ctypes.POINTER(tdp._Problem), ctypes.POINTER(ctypes.c_void_p)]
    assert lib.tdp_plan_create(ctypes.byref(pr), ctypes.byref(h)) == 3
    assert lib.tdp_plan_create(None, ctypes.byref(h)) == 1
    lib.tdp_blend.argtypes = [ctypes.c_void_p] * 4
    assert lib.tdp_blend(None, None, None, None) == 1
    lib.tdp_split.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int32] + [ctypes.c_void_p] * 3
    assert lib.tdp_split(None, None, None, None, 1, None, None, None) == 1
    lib.tdp_pos_bounds.argtypes = [ctypes.c_void_p] * 5
    assert lib.tdp_pos_bounds(None, None, None, None, None) == 1


@no_gpu_only
def test_host_validation_before_launch(tdp):
    """Argument errors return a status without touching CUDA (runs without a GPU)."""
    lib = ctypes.CDLL(tdp.LIB_PATH)
    plan = tdp.tdp_plan_create(1, 3, 8, 12, 16, "f32", (1, 2, 2), (0, 2, 2))
    vp = ctypes.c_void_p
    lib.tdp_split.argtypes = [vp, vp, vp, vp, ctypes.c_int32, vp, vp, vp]
    lib.tdp_pos_bounds.argtypes = [vp, vp, vp, vp, vp]
    lib.tdp_blend.argtypes = [vp, vp, vp, vp]
    lib.tdp_norm_filter.argtypes = [vp, vp, ctypes.c_int32, vp, vp, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp]
    lib.tdp_cond_blend.argtypes = [vp, ctypes.c_int32, ctypes.c_int32, vp, vp, vp, vp]
    lib.tdp_tile_mean.argtypes = [vp, ctypes.c_int64, vp, vp, vp]
    # positions without an output for them, and normalising without mn
    assert lib.tdp_split(plan.handle, 16, 8, 16, 1, 16, None, None) == 1
    assert lib.tdp_split(plan.handle, 16, 8, None, 1, 16, 8, None) == 1
    # misaligned latent pointer (never dereferenced: refused on the host)
    assert lib.tdp_split(plan.handle, 24, None, None, 1, 16, None, None) == 4
    assert lib.tdp_pos_bounds(plan.handle, None, 16, 16, None) == 1
    assert lib.tdp_pos_bounds(plan.handle, 4, 16, 16, None) == 4
    assert lib.tdp_blend(plan.handle, 16, 40, None) == 4
    assert lib.tdp_blend(plan.handle, None, 16, None) == 1
    assert lib.tdp_norm_filter(plan.handle, None, -1, 16, 16, 1, None, None, 16, None, None, None, None) == 1
    assert lib.tdp_norm_filter(plan.handle, 8, 4, 16, 16, 1, 16, 16, 16, 16, 12, None, None) == 4
    assert lib.tdp_norm_filter(plan.handle, 8, 4, 16, 16, 1, 16, 16, 16, 16, 16, 6, None) == 4   # slot
    assert lib.tdp_cond_blend(plan.handle, 4, 0, 16, 16, 16, None) == 1                           # ncap < 1
    assert lib.tdp_cond_blend(plan.handle, 4, 4, 24, 16, 16, None) == 4                           # Ycond
    assert lib.tdp_cond_blend(plan.handle, 4, 4, 16, None, 16, None) == 1
    assert lib.tdp_tile_mean(plan.handle, 3, 16, 16, None) == 4                                   # 12 bytes
    assert lib.tdp_tile_mean(plan.handle, 8, 16, 40, None) == 4
    assert lib.tdp_tile_mean(plan.handle, -1, 16, 16, None) == 1
    # tdp_split_filter(plan, X, P, K, N, normalize, Y, Q, mn, mx, keep, idx, count, kcount, Kout, slot, s)
    i32 = ctypes.c_int32
    lib.tdp_split_filter.argtypes = [vp, vp, vp, vp, i32, i32] + [vp] * 11
    ok = dict(X=16, P=8, K=8, N=4, Y=16, Q=8, mn=16, mx=16, keep=16, idx=16, count=16, kcount=16, Kout=16)

    def sf(**kw):
        a = dict(ok, **kw)
        return lib.tdp_split_filter(plan.handle, a["X"], a["P"], a["K"], a["N"], 1, a["Y"], a["Q"], a["mn"],
                                    a["mx"], a["keep"], a["idx"], a["count"], a["kcount"], a["Kout"],
                                    a.get("slot"), None)
    assert sf(P=None) == 1 and sf(Q=None) == 1                 # the bounds need positions
    assert sf(N=-1) == 1
    assert sf(mx=None) == 1 and sf(count=None) == 1 and sf(Kout=None) == 1
    assert sf(X=24) == 4 and sf(K=12) == 4 and sf(slot=6) == 4 and sf(Q=4) == 4
    assert lib.tdp_split_filter(None, 16, 8, 8, 4, 1, 16, 8, 16, 16, 16, 16, 16, 16, 16, None, None) == 1


def test_binding_refuses_wrong_sizes_on_host(tdp):
    torch = pytest.importorskip("torch")
    plan = tdp.tdp_plan_create(1, 3, 8, 12, 16, "f32", (1, 2, 2), (0, 2, 2))
    with pytest.raises(ValueError):
        tdp.tdp_blend(plan, torch.zeros(10), torch.zeros(10))   # CPU tensors are refused


@no_gpu_only
def test_zero_batch_is_a_no_op(tdp):
    lib = ctypes.CDLL(tdp.LIB_PATH)
    plan = tdp.tdp_plan_create(0, 3, 8, 12, 16, "f32", (1, 2, 2), (0, 2, 2))
    vp = ctypes.c_void_p
    lib.tdp_blend.argtypes = [vp, vp, vp, vp]
    assert lib.tdp_blend(plan.handle, None, None, None) == 0


def test_threads_share_a_plan_and_keep_their_own_error_detail(tdp):
    """A plan is immutable and usable from any host thread; the error detail is per thread."""
    import threading
    plan = tdp.tdp_plan_create(1, 16, 32, 48, 128, "bf16", (1, 2, 2), (0, 8, 8))
    ref = tdp.tdp_plan_info(plan)
    errors = []

    def worker(i):
        try:
            for _ in range(200):
                n, tot, boxes, offs = tdp.tdp_plan_info(plan)
                assert n == ref[0] and tot == ref[1]
                assert np.array_equal(boxes, ref[2]) and np.array_equal(offs, ref[3])
                assert list(tdp.tdp_rank_tiles(plan, i % 4, 4)) == list(range(i % 4, n, 4))
                bad = dict(C=6) if i % 2 else dict(num_tiles=(1, 99, 1))
                with pytest.raises(tdp.TdpError) as ei:
                    tdp.tdp_plan_create(1, 3, 8, 12, bad.get("C", 16), "bf16", bad.get("num_tiles", (1, 2, 2)),
                                        (0, 2, 2))
                detail = tdp.tdp_last_error_detail()
                assert ("multiple of 16" in detail) if i % 2 else ("multiple of 16" not in detail and detail)
                assert ei.value.status == (4 if i % 2 else 2)
        except Exception as e:        # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:3]


def test_cond_records_size_and_refusals(tdp):
    """The records' size follows the documented layout (G records of ceil4(26 + 8 nt) ints,
    then the deal, 8 tokens per record, 8 G ints of per-token info, B N nt ints of per-token
    lists and the deal's tables, 32 ceil(B N / 32) + 16 ints); shapes the records do not take,
    and bad arguments, are refused on the host."""
    lib = ctypes.CDLL(tdp.LIB_PATH)
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.tdp_cond_records_size.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int64)]
    lib.tdp_cond_records.argtypes = [vp, i32, i32, vp, vp, vp]
    lib.tdp_cond_blend_records.argtypes = [vp, i32, i32, vp, vp, vp, vp]
    for wl in wk.WORKLOADS:
        plan = tdp.tdp_plan_create(wl.B, wl.F, wl.H, wl.W, wl.C, wl.dtype, wl.num_tiles, wl.overlap)
        G = wl.B * ((wl.n_cond + 7) // 8)
        rec = (26 + 8 * plan.n_tiles + 3) // 4 * 4
        P = (wl.B * wl.n_cond + 31) // 32
        assert tdp.tdp_cond_records_size(plan, wl.n_cond) == \
            G * rec + 16 * G + wl.B * wl.n_cond * plan.n_tiles + 32 * P + 16
    plan = tdp.tdp_plan_create(1, 3, 8, 12, 16, "f32", (1, 2, 2), (0, 2, 2))
    n = ctypes.c_int64(-1)
    assert lib.tdp_cond_records_size(plan.handle, 0, ctypes.byref(n)) == 0 and n.value == 0
    assert lib.tdp_cond_records_size(plan.handle, -1, ctypes.byref(n)) == 1
    assert lib.tdp_cond_records_size(None, 4, ctypes.byref(n)) == 1
    # N = 0: nothing to do, nothing read
    assert lib.tdp_cond_records(plan.handle, 0, 1, None, None, None) == 0
    assert lib.tdp_cond_blend_records(plan.handle, 0, 1, None, None, None, None) == 0
    assert lib.tdp_cond_blend_records(plan.handle, 4, 0, None, None, None, None) == 1      # ncap < 1
    assert lib.tdp_cond_records(plan.handle, 4, 0, None, None, None) == 1          # ncap < 1
    assert lib.tdp_cond_records(plan.handle, 4, 1, None, None, None) == 1          # null slot
    # 257 tiles or more: beyond the records (tdp_cond_blend takes them)
    big = tdp.tdp_plan_create(1, 2, 48, 52, 8, "bf16", (1, 16, 17), (0, 1, 1))
    assert big.n_tiles > 256
    assert lib.tdp_cond_records_size(big.handle, 8, ctypes.byref(n)) == 5
    assert lib.tdp_cond_records(big.handle, 8, 1, None, None, None) == 5
    assert lib.tdp_cond_blend_records(big.handle, 8, 1, None, None, None, None) == 5


@no_gpu_only
def test_cond_records_alignment_refused_on_host(tdp):
    lib = ctypes.CDLL(tdp.LIB_PATH)
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.tdp_cond_records.argtypes = [vp, i32, i32, vp, vp, vp]
    lib.tdp_cond_blend_records.argtypes = [vp, i32, i32, vp, vp, vp, vp]
    plan = tdp.tdp_plan_create(1, 3, 8, 12, 16, "f32", (1, 2, 2), (0, 2, 2))
    assert lib.tdp_cond_records(plan.handle, 4, 1, 16, 8, None) == 4               # recs not 16-byte aligned
    assert lib.tdp_cond_records(plan.handle, 4, 1, 6, 16, None) == 4               # slot not 4-byte aligned
    assert lib.tdp_cond_blend_records(plan.handle, 4, 1, 8, 16, 16, None) == 4
    assert lib.tdp_cond_blend_records(plan.handle, 4, 1, 16, 24, 16, None) == 4
    assert lib.tdp_cond_blend_records(plan.handle, 4, 1, 16, 16, None, None) == 1
