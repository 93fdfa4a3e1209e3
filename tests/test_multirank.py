"""The benchmark's multi-rank logic (replicas, max time over ranks, rank 0
prints) on world_size-2 gloo process groups on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slow = bench.max_over_ranks(10.0 + 5.0 * rank)  # rank 1 is the slow one
        ws, r, local = bench._dist()

        class A:
            steps, warmup = 1, 1
        # the reference arm runs on rank 0 only; the other ranks return nothing
        ref = bench.run_reference(A) if rank == 1 else "skipped"
        q.put((rank, slow, ws, r, ref))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rank0_only_on_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {o[0]: o for o in out}
    assert by_rank[0][1] == 15.0 and by_rank[1][1] == 15.0   # both see the slowest rank
    assert by_rank[0][2] == 2 and by_rank[1][3] == 1
    assert by_rank[1][4] is None


def test_job_throughput_is_whole_job():
    import bench
    # two replicas of 100 GFLOP per step, 10 steps, slowest rank 20 ms in total
    assert bench.job_throughput(2, 100e9, 10, 20.0) == pytest.approx(100.0)
    assert bench.max_over_ranks(3.5) == 3.5  # no process group: unchanged
