"""Host logic of the multi-rank benchmark, run as two gloo ranks on the CPU: the tensors are
split across ranks with no overlap and no gap (the path needs no data exchange), the
timing reduction takes the slowest rank, and the reference arm does its work on rank 0
only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, n_tensors, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)  # CPU ranks, even on a GPU host
    r, w = bench._dist()
    assert (r, w) == (rank, world)
    lo, hi = bench.shard(n_tensors, rank, world)
    slowest = bench._max_over_ranks(10.0 + rank, world)
    ran = []

    class Args:
        warmup, steps, gpus = 0, 1, world

    # the reference arm: rank 0 would run the oracle; the others must return at once
    if rank != 0:
        bench.run_reference(Args, None)
        ran.append("returned")
    q.put((rank, lo, hi, slowest, ran))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("n_tensors", [24, 7, 1])
def test_two_rank_shards_cover_every_tensor_once(n_tensors):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n_tensors, q))
             for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    covered = []
    for rank, lo, hi, slowest, ran in got:
        covered.extend(range(lo, hi))
        assert slowest == 11.0  # max over ranks, not the rank's own time
        if rank != 0:
            assert ran == ["returned"]
    assert sorted(covered) == list(range(n_tensors))
    sizes = [hi - lo for _, lo, hi, _, _ in got]
    assert max(sizes) - min(sizes) <= 1
