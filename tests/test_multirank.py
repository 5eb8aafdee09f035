"""Host-side logic of the multi-GPU bench on CPU: two gloo ranks, each with its own seeded batch
(weak scaling), gathered per-rank times, whole-job throughput over the slowest rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from state_space_sequence_gb300 import inputs


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    assert (r, w) == (rank, world)
    wl = inputs.make_dlr(2, 3, 4, 16, seed=bench.rank_seed(1, rank))
    # a fake per-rank time: rank 1 is slower
    t = torch.tensor([1.0 + rank], dtype=torch.float64)
    gathered = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(gathered, t)
    value, tmax = bench.aggregate([float(g.item()) for g in gathered], units_per_rank=96)
    q.put((rank, float(wl.u.sum()), value, tmax))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_batches_and_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    (_, s0, v0, t0), (_, s1, v1, t1) = res
    assert s0 != s1                      # each rank drew its own batch
    assert t0 == t1 == 2.0               # max over ranks
    assert v0 == v1 == pytest.approx(96 * 2 / 2.0)


def test_aggregate_single_rank():
    v, t = bench.aggregate([0.5], 100)
    assert t == 0.5 and v == 200
