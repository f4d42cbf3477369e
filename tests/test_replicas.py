"""The multi-GPU path is replicas only: each rank runs its own (batch, KV head) rows and the bench reduces the
timings (max) and throughputs (sum) over ranks. Its host logic runs here as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, wsz, dist = bench._dist_init(world)
    try:
        bench._barrier(dist)
        out.put((r, wsz, bench._max_over_ranks(dist, float(r + 1)), bench._sum_over_ranks(dist, float(r + 1))))
        bench._barrier(dist)
    finally:
        dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo path is the host without CUDA")
def test_two_gloo_ranks_reduce_timings_and_throughputs():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[:2] for x in res] == [(0, 2), (1, 2)]
    assert all(x[2] == 2.0 and x[3] == 3.0 for x in res)   # max over ranks of r+1, sum over ranks
