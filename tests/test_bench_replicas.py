"""The multi-GPU path is replicas only (every (batch, head) problem is
independent; no data-path collective).  What the N>1 run adds is the timing
aggregation: the slowest rank's time and the sum of all ranks' work.  Checked
here with two gloo ranks on the CPU."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = 10.0 + 5.0 * rank          # rank 1 is the slowest
    flops_local = 1e12 * (rank + 1)
    bench.barrier(dist)
    ms, tflops = bench.aggregate(ms_local, flops_local, dist, torch.device("cpu"))
    out[rank] = (ms, tflops)
    dist.destroy_process_group()


def test_replica_aggregation_gloo_two_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        ms, tflops = res[r]
        assert ms == 15.0                          # max over ranks
        assert tflops == pytest.approx(3e12 / 15e-3 / 1e12)  # total work / slowest time


def test_single_process_aggregation():
    import bench
    ms, tflops = bench.aggregate(20.0, 2e12, None, torch.device("cpu"))
    assert ms == 20.0 and tflops == pytest.approx(100.0)
