"""The multi-GPU path of the benchmark is N independent replicas (the routed-expert path has no
exchange step of its own); what crosses ranks is the barrier around the timed region and the
max-over-ranks of the elapsed time, and the reference arm runs on rank 0 only.  Checked here
with world_size-2 gloo process groups on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    # the slowest rank sets the value every rank reports
    m = bench.max_over_ranks(10.0 + rank * 5.0, world, torch.device("cpu"))
    dist.barrier()
    # the reference arm: ranks other than 0 leave without work
    ran = []

    class A:
        steps, warmup = 1, 0

    if rank != 0:
        bench.run_reference(A, rank, world)
        ran.append("skipped")
    out.put((rank, m, ran))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_and_rank0_only_reference():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[1][2] == ["skipped"]


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
