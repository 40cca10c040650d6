"""The bench's multi-rank host logic on CPU with world size 2 (gloo): the
timing is the maximum over ranks, throughput counts every rank's units, and
under torchrun only rank 0 prints the reference arm's line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank 0 is slower on the first value, rank 1 on the second
        got = bench.max_over_ranks([10.0 + rank, 5.0 - rank], "cpu", world)
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_timing_is_the_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res[0] == res[1] == [11.0, 5.0]


def test_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 64 sequences per rank and step, 2 ranks, 10 steps in 2 ms
    assert bench.job_throughput(64, 2, 10, 2.0) == pytest.approx(640000.0)
    assert bench.max_over_ranks([3.0, 1.5], "cpu", 1) == [3.0, 1.5]


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny_fp32", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
