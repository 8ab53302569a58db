"""CPU checks of the benchmark's host logic: the cross-rank reduction (two gloo
ranks), the byte and FLOP accounting, and the oracle reference arm."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from gated_delta_net_gb300 import workloads as W  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [0.5, 2.0][rank]
    t = bench.reduce_max(elapsed)
    q.put((rank, t, bench.job_throughput(1000, 10, t, world)))
    dist.destroy_process_group()


def test_two_rank_max_reduction_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, t, v in out:
        assert t == 2.0
        assert v == pytest.approx(1000 * 2 * 10 / 2.0)


def test_reduce_max_without_process_group():
    assert bench.reduce_max(3.5) == 3.5


def test_verify_bytes_throughput_point():
    tb = W.serving_target()
    # per request: S0 + 128 nodes x (q,k + v + g,beta + o + parent + depth + 4 mask words)
    per_req = 32 * 128 * 128 * 4 + 128 * (2 * 16 * 128 * 2 + 32 * 128 * 2 + 32 * 8 + 32 * 128 * 2 + 4 + 4 + 16)
    assert bench.verify_bytes(tb) == 64 * per_req + 4 * 65


def test_verify_flops_chain_closed_form():
    tb = W.custom(1, [W.chain_tree(10)], n_k_heads=1, n_v_heads=1, d=16)
    P = sum(range(1, 11))
    assert bench.verify_flops(tb) == 4 * 10 * 16 * 16 + 2 * 16 * (4 * P - 2 * 10)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--batch", "2", "--tree-size", "16",
                        "--ref-seconds", "0.05"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["unit"] == bench.UNIT and line["higher_is_better"] is True
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_clock_summary_keeps_only_the_timed_window():
    import datetime
    import bench

    def line(sec, mhz, thermal="Not Active"):
        t = datetime.datetime(2026, 1, 1, 12, 0, sec, 500000).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{t}, {mhz}, 2070, 900.1, 0x0, Not Active, {thermal}, Not Active, Not Active"

    lines = [line(0, 1000), line(1, 2070), line(2, 2000, "Active"), line(3, 2070), line(9, 500)]
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 1).timestamp()
    s = bench.summarize_clocks(lines, t0, t0 + 3)
    assert s["window"] == "timed region" and s["samples"] == 3
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["hw_thermal_slowdown"]
    s = bench.summarize_clocks(lines, t0 + 100, t0 + 101)
    assert s["window"] == "around the timed region" and s["samples"] == 5
    assert bench.summarize_clocks([]) is None


def test_source_hash_ignores_comments(tmp_path, monkeypatch):
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "a.cu").write_text("int x = 1;  // one\n\n// note\nint y;\n")
    h1 = bench.source_sha(["a.cu"])
    (tmp_path / "a.cu").write_text("int x = 1;  // changed words\n// another note\nint y;\n")
    assert bench.source_sha(["a.cu"]) == h1
    (tmp_path / "a.cu").write_text("int x = 2;\nint y;\n")
    assert bench.source_sha(["a.cu"]) != h1


@pytest.mark.parametrize("depth,size,workload,kernel,commit", [
    (16, 128, "serving_b64_n128", "verify_tc", "commit_tc"),
    (16, 256, "serving_b64_n256", "verify_wide", "commit_tc"),
    (32, 128, "deep_b64_n128_d32", "verify_wide", "commit_tc"),
    (64, 128, "deep_b64_n128_d64", "verify_wide", "commit_simt"),
    (0, 128, "serving_b64_n128_nobound", "verify_simt", "commit_simt"),
])
def test_bench_workload_and_kernel(depth, size, workload, kernel, commit):
    import argparse
    args = argparse.Namespace(depth=depth, batch=64, tree_size=size)
    tb = bench.bench_workload(args)
    assert tb.name == workload
    assert bench.dominant_kernel(tb) == kernel
    assert bench.commit_kernel(tb) == commit
    assert tb.max_nodes == size
    # the declared depth bound holds for every tree, and deep workloads reach past 16
    depth_of = np.ones(tb.total_nodes, np.int64)
    for b in range(tb.batch):
        lo = int(tb.node_offsets[b])
        for i in range(int(tb.node_offsets[b + 1]) - lo):
            a = tb.parent[lo + i]
            depth_of[lo + i] = 1 if a < 0 else depth_of[lo + a] + 1
    if depth:
        assert depth_of.max() <= max(depth, 16)
    if depth > 16:
        assert depth_of.max() > 16


def test_traffic_entries_match_their_workloads():
    # every recorded capture names its workload and command, and a kernel's
    # entries are for distinct workloads
    with open(bench.TRAFFIC_FILE) as f:
        tr = json.load(f)
    for kernel, ents in tr.items():
        assert kernel in bench.KERNEL_SOURCES
        ents = ents if isinstance(ents, list) else [ents]
        names = [e["workload"] for e in ents]
        assert len(names) == len(set(names))
        for e in ents:
            assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
            assert e["command"].startswith("ncu ") and "--clock-control none" in e["command"]
