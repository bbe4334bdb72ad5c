"""Multi-rank bookkeeping of the benchmark on CPU (gloo, world size 2): each
rank runs its own replica of the matrix set (distinct seeds, no collective on
the data path); the reported time is the max over ranks and the value counts
every rank's work."""

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from matrix_optimizer_update_gb300 import workloads as wl
    from matrix_optimizer_update_gb300.inputs import make_matrix_set

    r, w, _ = bench.dist_env()
    assert (r, w) == (rank, world)
    # replicas draw different data
    toy = wl.get("toy")
    ms = make_matrix_set(toy, "cpu", seed_offset=bench.replica_seed_offset(rank))
    g0 = ms.G[:8].clone()
    gathered = [torch.zeros_like(g0) for _ in range(world)]
    dist.all_gather(gathered, g0)
    distinct = not torch.equal(gathered[0], gathered[1])
    # each rank "took" a different time; everyone must report the slowest
    t = bench.max_over_ranks(10.0 + rank, world)
    v = bench.aggregate(1e12, 4, world, t)
    out.put((rank, distinct, t, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, distinct, t, v in res:
        assert distinct
        assert t == 11.0
        assert v == pytest.approx(1e12 * 4 * 2 / 11.0 / 1e12)
