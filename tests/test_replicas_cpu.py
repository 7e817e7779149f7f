"""The multi-GPU path of the benchmark is independent replicas (the decode step does not shard):
the job's time is the slowest rank's, its throughput the sum over ranks.  Checked here on CPU with
two gloo ranks, and that only rank 0 of the reference arm prints."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

import bench

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(dist, torch, 4.0 + rank, "cpu")   # rank r took 4 + r ms per token
        q.put((rank, slowest, bench.replica_throughput(world, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_sum_replicas():
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [5.0, 5.0]              # both ranks see the max over ranks
    assert out[0][2] == pytest.approx(2 * 1e3 / 5.0)      # 2 replicas, 5 ms per token each


def test_single_process_is_its_own_max():
    assert bench.max_over_ranks(None, torch, 3.25, "cpu") == 3.25
    assert bench.replica_throughput(1, 4.0) == 250.0


def test_reference_arm_prints_on_rank_zero_only():
    class A:
        steps, warmup = 1, 0
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A, 1, 2)
    assert buf.getvalue() == ""
