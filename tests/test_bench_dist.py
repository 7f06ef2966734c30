"""The benchmark's multi-process path (one replica per GPU under torchrun):
barrier, max-over-ranks timing and whole-job sums, on two gloo ranks on the
CPU.  No GPU is involved."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    t_max = bench.max_over_ranks(w, 1.0 + rank)          # per-rank elapsed seconds
    total = bench.sum_over_ranks(w, 1000.0 * (rank + 1))  # per-rank values processed
    q.put((rank, t_max, total))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_replicas_reduce_timing_and_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(0, 2.0, 3000.0), (1, 2.0, 3000.0)]
