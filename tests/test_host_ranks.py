"""The bench's N > 1 host logic on CPU: two ``gloo`` ranks (world size 2).

Under torchrun each rank runs an independent replica of the workload; the job's time is
the slowest rank's, and its rate counts the units of every rank.  The reference arm runs on
rank 0 only; the other ranks leave without work.
"""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's step time and end-to-end time; the slowest of each must win on every rank
        mine = [1.0 + rank, 5.0 - 2 * rank]
        got = bench.max_over_ranks(mine, torch.device("cpu"))
        dist.barrier()
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res[0] == res[1] == [2.0, 5.0]


def test_single_rank_keeps_its_own_times():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([0.25, 3], "cpu") == [0.25, 3.0]


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas x 10 steps x 1,000 tokens in 4 s (the slowest rank's time)
    assert bench.job_throughput(2, 10, 1000, 4.0) == 5000.0
    assert bench.job_throughput(1, 10, 1000, 4.0) == 2500.0


@pytest.mark.parametrize("rank", [1, 3])
def test_reference_arm_other_ranks_exit_without_work(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="4", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank_zero_prints_one_json_line():
    # rank 0's reference line is one JSON object with the contract's keys
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "1", "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
