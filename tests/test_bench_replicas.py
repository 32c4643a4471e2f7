"""The multi-GPU path of the benchmark is replicas only (the decode step shards by
request with no exchange step): each rank times its own steps and the job's
throughput is all ranks' steps over the slowest rank's time.  Checked with two
gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [80.0, 100.0][rank]            # rank 1 is the slower replica
    value, ms = bench.aggregate_replicas(local, steps=20, pg=dist, device="cpu")
    q.put((rank, value, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
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
    for rank, value, ms in out:
        assert ms == pytest.approx(100.0 / 20)
        assert value == pytest.approx(2 * 20 / 0.1)


def test_single_process_has_no_collective():
    value, ms = bench.aggregate_replicas(50.0, steps=10)
    assert value == pytest.approx(10 / 0.05) and ms == pytest.approx(5.0)
