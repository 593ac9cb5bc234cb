"""bench.py host logic on CPU: FLOP accounting against brute force, the
reference-arm JSON line, and the multi-rank reduction under gloo."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def brute_pairs(seg_row, exclude_last=False):
    N = len(seg_row)
    last = seg_row[-1]
    n = 0
    for i in range(N):
        for j in range(i + 1):
            if seg_row[i] == seg_row[j] and not (exclude_last and seg_row[i] == last):
                n += 1
    return n


def test_visible_pairs_match_brute_force():
    w = synth.custom(2, 2, 1, 256, 64, [[1, 100, 155], [7, 249]])
    assert bench.visible_pairs_per_head(w) == brute_pairs(w.seg[0]) + brute_pairs(w.seg[1])
    w.pad = [155, 0]  # first row's last segment is padding
    assert bench.visible_pairs_per_head(w) == brute_pairs(w.seg[0], True) + brute_pairs(w.seg[1])
    assert bench.useful_flops(w) == 14 * 64 * bench.visible_pairs_per_head(w) * 2


def test_executed_tiles_match_brute_force():
    w = synth.custom(1, 1, 1, 640, 64, [[100, 300, 28, 212]])
    T = 5
    seg = w.seg[0]
    n = 0
    for tq in range(T):
        for tk in range(tq + 1):
            a = set(seg[tq * 128:(tq + 1) * 128].tolist())
            b = set(seg[tk * 128:(tk + 1) * 128].tolist())
            n += bool(a & b)  # contiguous runs: range overlap == shared id
    assert bench.executed_tile_pairs(w) == n
    assert bench.executed_tile_pairs(synth.custom(1, 1, 1, 512, 64, [[512]])) == 10


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny_3seg", "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOPS"
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["higher_is_better"] is True


def test_reference_arm_non_zero_rank_is_silent():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny_3seg", "--steps", "1"], capture_output=True, text=True, timeout=120, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier()
    m = bench.reduce_max(1.5 + rank)  # each rank's "step time"
    seed = bench.replica_seed(1004, rank)
    q.put((rank, m, seed))
    dist.destroy_process_group()


def test_multi_rank_reduction_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [m for _, m, _ in res] == [2.5, 2.5]           # max over ranks, seen by every rank
    assert res[0][2] != res[1][2]                         # independent replica inputs per rank


def test_lce_extra_reports_failure_instead_of_raising():
    """The cross-entropy measurement runs in a child process; without a GPU
    the child fails and the extra reports it as an error entry."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import bench
    r = bench.lce_extra()
    assert set(r) == {"error"} and r["error"].startswith("exit ")
