"""The multi-rank host logic of bench.py on CPU: two gloo ranks (one process
each, as torchrun starts them) reduce their timings and token counts the way
the benchmark does (time = max over ranks, tokens = sum over ranks, so
throughput = all ranks' tokens / the slowest rank's time), meet at barriers,
and only rank 0 runs the CPU reference arm."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w = bench.dist_setup(world)
    assert (r, w) == (rank, world) and dist.get_backend() == "gloo"
    t_step = 1.0 + rank                    # rank 1 is the slower one
    tokens = 4096 * (rank + 1)
    bench.barrier(w)
    t_max = bench.max_over_ranks(t_step, w)
    total = bench.sum_over_ranks(tokens, w)
    value = total / t_max
    # the reference arm: every rank but 0 returns at once, without work
    out = None
    if rank != 0:
        out = bench.run_reference(None, r, w)
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((rank, t_max, total, value, out))


@pytest.mark.timeout(300)
def test_two_gloo_ranks_reduce_like_the_benchmark():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, total, value, out in res:
        assert t_max == 2.0                 # max over ranks
        assert total == 4096 + 8192         # sum over ranks
        assert value == pytest.approx(12288 / 2.0)
        assert out is None
