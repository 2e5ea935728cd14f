"""The N-GPU bench path on CPU: world_size-2 gloo ranks run independent
replicas; the job time is the slowest rank's and the value counts every
rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    total_ms = [30.0, 50.0][rank]  # rank 1 is the slower replica
    ms, value = bench.replica_throughput(total_ms, steps=10, tokens_per_replica=4096,
                                         world_size=world, device="cpu")
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_max_time_and_sum_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, ms, value in res:
        assert ms == pytest.approx(5.0)               # 50 ms / 10 steps, the slower rank
        assert value == pytest.approx(2 * 4096 / 5e-3)


def test_single_replica_needs_no_process_group():
    import bench
    ms, value = bench.replica_throughput(12.0, steps=4, tokens_per_replica=100, world_size=1)
    assert ms == 3.0 and value == pytest.approx(100 / 3e-3)
