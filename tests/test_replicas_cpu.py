"""The multi-GPU path is N independent replicas (the layer has no cross-GPU
exchange).  bench.py's whole-job aggregation -- slowest rank's times, tokens
of all ranks over that time -- checked with two gloo ranks on the CPU."""
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


def _rank(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took (r + 1) * 0.1 s of device time and (r + 1) * 0.2 s end to end
        dev_s, e2e_s, value = bench.aggregate_replicas(0.1 * (rank + 1), 0.2 * (rank + 1), 1000, world,
                                                       torch.device("cpu"))
        queue.put((rank, dev_s, e2e_s, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_aggregate_max_time_and_all_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, queue)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(queue.get(timeout=10) for _ in range(world))
    for rank, dev_s, e2e_s, value in got:
        assert dev_s == pytest.approx(0.2)   # the slower rank
        assert e2e_s == pytest.approx(0.4)
        assert value == pytest.approx(2 * 1000 / 0.2)


def test_single_replica_needs_no_process_group():
    import bench
    dev_s, e2e_s, value = bench.aggregate_replicas(0.5, 0.7, 100, 1, torch.device("cpu"))
    assert (dev_s, e2e_s, value) == (0.5, 0.7, 200.0)
