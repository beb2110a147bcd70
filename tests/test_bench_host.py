"""bench.py on the host: the reference arm's JSON line (it runs the CPU oracle and needs
no GPU), the algorithmic-byte formulas, and the parser of the committed DRAM-traffic file."""
import json
import os
import subprocess
import sys

import numpy as np

import oracle
import workloads as wk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_line_keeps_the_contract():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, "the bench prints exactly one JSON line"
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("tiny:") and "host CPU" in d["config"]["l2"]


def test_reference_arm_rejects_short_warmup():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "2"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode != 0


def test_algorithmic_bytes_of_the_large_workload():
    """Each call's minimum bytes, recounted here from the sizes of what it must read and write."""
    wl = wk.by_name("large")
    box, off = oracle.plan(oracle.problem_of(wl))
    nt, tot = box.shape[0], int(off[-1])
    kept = 220890
    ab = bench.algorithmic_bytes(wl, tot, nt, kept)
    latent = wl.B * wl.tokens * wl.C * 2                       # bf16 latent, read or written once
    tiles = wl.B * tot * wl.C * 2                              # every tile token once
    pos_in, pos_out = wl.B * wl.tokens * 3 * 8, wl.B * tot * 3 * 8   # [B,3,T,2] int32 and its tiles
    assert ab["split"] == latent + tiles + pos_in + pos_out
    assert ab["blend"] == tiles + latent
    assert ab["bounds"] == pos_in + 2 * nt * wl.B * 3 * 4
    N = wl.n_cond
    assert ab["filter"] == wl.B * N * 24 + nt * wl.B * N * 5 + nt * wl.B * 4 + wl.B * N * 4 + kept * 24
    assert ab["step"] == ab["split"] + ab["filter"] + ab["blend"] + 2 * nt * wl.B * 3 * 4
    assert abs(ab["blend"] / 1e6 - 1672.7) < 0.1 and abs(ab["split"] / 1e6 - 1829.6) < 0.1


def test_traffic_file_parser(tmp_path, monkeypatch):
    rows = {k: bench.kernel_source_hash(v) for k, v in bench.KERNEL_SOURCES.items()}
    text = "# comment line\n" + "\n".join(
        f"{k} {h} {100 + i} {10 + i} 5 0" for i, (k, h) in enumerate(sorted(rows.items()))) + "\n"
    f = tmp_path / "dram_traffic_large.txt"
    f.write_text(text)
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    order = sorted(rows)
    expect = {k: 100 + i + 10 + i for i, k in enumerate(order)}
    assert bench.profiled_traffic("tdp_blend") == expect["tdp_blend_kernel"]
    assert bench.profiled_traffic("tdp_split_filter") == sum(
        expect[k] for k in ("tdp_bounds_init_kernel", "tdp_bounds_kernel", "tdp_split_filter_kernel"))
    # a kernel whose sources changed since the capture has no traffic figure
    f.write_text(text.replace(rows["tdp_blend_kernel"], "0" * 16))
    assert bench.profiled_traffic("tdp_blend") is None
    f.write_text("# nothing captured\n")
    assert bench.profiled_traffic("tdp_split_filter") is None
    # another workload has no capture of its own: no figure, not the large workload's
    f.write_text(text)
    assert bench.profiled_traffic("tdp_blend", "large") == expect["tdp_blend_kernel"]
    assert bench.profiled_traffic("tdp_blend", "temporal") is None


def test_committed_traffic_files_parse():
    """Every committed traffic file is named for a workload, and every line of it has a kernel
    the bench knows and integer fields."""
    import glob
    names = {w.name for w in bench.wk.WORKLOADS}
    files = glob.glob(os.path.join(bench.PROFILE_DIR, "dram_traffic_*.txt"))
    assert files
    for path in files:
        assert os.path.basename(path)[len("dram_traffic_"):-len(".txt")] in names
        lines = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
        assert lines
        for parts in lines:
            assert parts[0] in bench.KERNEL_SOURCES and len(parts[1]) == 16
            assert all(np.int64(int(x)) >= 0 for x in parts[2:6])


def test_reference_arm_under_torchrun_prints_one_line():
    """Launched as the driver launches N > 1 (torchrun, one process per rank): rank 0 alone
    runs the oracle and prints; the other ranks exit 0 without work."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port),
                        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    assert json.loads(lines[0])["impl"] == "reference"
