"""Host-side logic of bench.py, on CPU: the multi-rank reduction (world size
2 over gloo) and the reference arm's JSON line on the tiny workload."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    ms, e2e, emitted = bench.combine_ranks(10.0 + rank, 20.0 - rank, 100.0 * (rank + 1), world, "cpu")
    q.put((rank, ms, e2e, emitted))
    dist.destroy_process_group()


def test_combine_ranks_max_time_sum_tokens_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, e2e, emitted in res:
        assert ms == 11.0 and e2e == 20.0 and emitted == 300.0


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "cfg0",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "requests/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == (os.cpu_count() or 1)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["steps"] == 3


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "cfg0",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_draft_steps_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "draft_cfg0", "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"].startswith("draft-step") and line["value"] > 0
    assert "3 greedy draft steps" in line["cpu_baseline"]["sample"]


def test_algorithmic_counts():
    sys.path.insert(0, ROOT)
    import bench
    import numpy as np
    w = bench.workloads()["draft_cfg1_D3"]
    a = bench.algorithmic(w, np.zeros(w.B, np.int64), draft=True)
    assert a["w_bytes"] == 3 * 129280 * 7168 * 2 and a["calls"] == 3 and a["kv_bytes"] == 0
    assert a["lm_flops"] == 2.0 * 32 * 7168 * 129280 * 3
    v = bench.workloads()["cfg1_D3"]
    ctx = np.array([512] * v.B, np.int64)
    b = bench.algorithmic(v, ctx)
    assert b["kv_bytes"] == v.B * (512 + 4) * 576 * 2 and b["calls"] == 1


def test_reference_arm_tree_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tree_cfg0", "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0


def test_tree_path_lengths():
    sys.path.insert(0, ROOT)
    import bench
    w = bench.workloads()["tree_cfg1_D15"]
    pl = bench.path_lengths(w)
    assert list(pl[0]) == [1, 2, 2, 2, 3, 3, 3, 3, 3, 3, 4, 4, 4, 4, 4, 4]
    v = bench.workloads()["cfg1_D3"]
    assert (bench.path_lengths(v) == [1, 2, 3, 4]).all()


def test_traffic_scaled_and_dropped_when_the_kernel_changes():
    sys.path.insert(0, ROOT)
    import bench
    files = bench.KERNEL_SOURCES["lm_head"]
    good = bench.source_digest(files)
    saved = dict(bench.TRAFFIC)
    try:
        bench.TRAFFIC["w"] = {"lm_head": (10.0, "vocabulary rows", files, good, "capture X")}
        t, note = bench.traffic_of("w", "lm_head", 3)
        assert t == 30.0 and "capture X" in note
        bench.TRAFFIC["w"] = {"lm_head": (10.0, "vocabulary rows", files, "0" * 16, "capture X")}
        t, note = bench.traffic_of("w", "lm_head", 3)
        assert t is None and "changed" in note
        assert bench.traffic_of("w", "attention", 3)[0] is None
    finally:
        bench.TRAFFIC.clear()
        bench.TRAFFIC.update(saved)


def test_workload_config_names_no_run_options():
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    cfg = bench.config_of(bench.workloads()["cfg3"], argparse.Namespace(no_graph=False, impl="gb300"))
    assert "cuda_graph" not in cfg and cfg["B"] == 256 and cfg["D"] == 3


def test_copy_in_pieces_matches_one_copy():
    """The end-to-end leg's copies in pieces give the same tensor as one copy,
    for sizes around and across the piece size, and leave views alone."""
    sys.path.insert(0, ROOT)
    import bench
    saved = bench.COPY_PIECE_BYTES
    try:
        bench.COPY_PIECE_BYTES = 64   # 16 float32 per piece
        g = torch.Generator().manual_seed(7)
        for n in (1, 15, 16, 17, 160, 161, 1000):
            src = torch.randn(n, generator=g)
            dst = torch.zeros(n)
            bench.copy_in_pieces(dst, src)
            assert torch.equal(dst, src), n
        src = torch.randn(7, 9, 5, generator=g)
        dst = torch.zeros(7, 9, 5)
        bench.copy_in_pieces(dst, src)
        assert torch.equal(dst, src)
        big = torch.zeros(10, 10)
        view = big[:, :3]                       # not contiguous: one plain copy
        bench.copy_in_pieces(view, torch.ones(10, 3))
        assert big[:, :3].eq(1).all() and big[:, 3:].eq(0).all()
    finally:
        bench.COPY_PIECE_BYTES = saved
