"""The multi-rank path of bench.py on CPU (gloo, world size 2).

The splice shards by request: every rank splices its own synthetic requests and no
data crosses ranks; the only collective is the max of the per-rank timings.  This
test runs that reduction and the job-throughput arithmetic on two gloo ranks.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out = bench.reduce_max_over_ranks([1.0 + rank, 10.0 - rank, 0.5], world, "cpu")
    q.put((rank, out, bench.rank_seed(7, rank), bench.dist_env()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_shard_seeds():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    for rank, out, seed, env in got:
        assert out == [2.0, 10.0, 0.5]
        assert env == (rank, 2, 0)
    assert got[0][2] != got[1][2]  # each rank draws its own requests


def test_job_value_counts_all_ranks():
    import bench
    assert bench.job_value(6768, 20, 2, 2.0) == 6768 * 20 * 2 / 2e-3
    assert bench.reduce_max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]
