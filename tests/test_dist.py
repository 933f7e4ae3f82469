"""The multi-rank host logic of bench.py on CPU: two gloo ranks join, agree on the slowest rank's step time and
report the whole-job throughput of per-rank replicas (no data-path collective exists in the prune step)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup(backend="gloo")
    assert (w, r, local) == (world, rank, rank)
    ms = 1.0 + rank                       # rank 1 is the slow one
    bench.dist_barrier(w)
    ms_max = bench.dist_max(ms, w)
    out[rank] = (ms_max, bench.job_throughput(1_000_000_000, ms_max, w))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        ms_max, gbs = out[r]
        assert ms_max == 2.0
        assert gbs == pytest.approx(2 * 1.0 / 2e-3, rel=1e-12)   # 2 ranks x 1 GB in 2 ms = 1000 GB/s
