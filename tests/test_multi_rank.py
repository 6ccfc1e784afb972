"""Multi-process logic of bench.py on CPU (gloo, world size 2).

The path runs as replicas: each rank computes the same workload on its own GPU
with no data exchange.  What needs checking is the host side: process-group
set-up from the torchrun environment, the max-over-ranks timing, the
whole-job aggregate, and that only rank 0 runs the reference arm.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # rank r "measured" (r + 1) ms for 1e12 FLOP
    ms, value = bench.aggregate(w, 1e12, float(rank + 1), torch.device("cpu"))
    out[rank] = (ms, value)
    # the reference arm: every rank but 0 returns without doing any work
    if rank != 0:
        class A:  # minimal argparse stand-in
            gpus, steps, warmup = world, 1, 0
        os.environ["RANK"] = str(rank)
        assert bench.run_reference(A(), bench.workload_of("c1")) is None
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replicas_take_max_time_and_sum_work():
    if torch.cuda.is_available():
        pytest.skip("gloo ranks on CPU; a machine with a GPU runs the single-GPU tests instead")
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    for r in range(2):
        ms, value = out[r]
        assert ms == 2.0                       # the slower rank sets the time
        assert abs(value - 2 * 1e12 / 2e-3 / 1e12) < 1e-9  # both ranks' work / max time
