"""The multi-rank path of bench.py on CPU: two gloo ranks reduce their
timings to the slowest rank's, the job's throughput counts every rank's
units, and under torchrun the reference arm prints from rank 0 only."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    # rank r took 10 + r ms for the device region and 20 - r for the end-to-end one
    out = b.max_over_ranks([10.0 + rank, 20.0 - rank], dist, torch.device("cpu"))
    dist.barrier()
    q.put((rank, out))
    dist.destroy_process_group()


def test_timings_reduce_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [11.0, 20.0]


def test_job_throughput_counts_every_rank():
    b = _bench()
    assert b.max_over_ranks([3.0, 4.5], None, None) == [3.0, 4.5]
    # 2048 tokens per rank and step, 5 steps, 2 ranks, 11 ms for the slowest rank
    assert b.job_throughput(2048, 5, 2, 11.0) == pytest.approx(2048 * 5 * 2 / 0.011)
    assert b.job_throughput(2048, 5, 1, 11.0) == pytest.approx(2048 * 5 / 0.011)


@pytest.mark.parametrize("rank", [1, 3])
def test_reference_arm_prints_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="4", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "4",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stderr[-500:]
    assert r.stdout.strip() == ""
