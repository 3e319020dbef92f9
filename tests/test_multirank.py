"""The N > 1 bench path on CPU: two gloo ranks each hold a batch of the same
shape with different values, and the reported time is the slowest rank's."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads
    seed = bench.rank_seed(rank)
    lengths = workloads.config_lengths(bench.WORKLOAD)
    # same lengths on every rank, different values
    pw = workloads.padded(lengths, 1, 8, seed)   # small H/D: shape logic only
    first = float(pw.q[0, 0, 0, 0])
    # a fake per-rank step time; the job's time is the maximum
    t = bench.max_over_ranks(10.0 + rank, dist)
    gathered = [None] * world
    dist.all_gather_object(gathered, (seed, lengths, first, t))
    if rank == 0:
        out.put(gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_weak_scaling_logic():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (s0, l0, f0, t0), (s1, l1, f1, t1) = res
    assert s0 != s1 and f0 != f1          # each rank its own values
    assert l0 == l1                        # same shape: per-GPU work fixed
    assert t0 == t1 == 11.0                # max over ranks on every rank
