"""The multi-replica timing of bench.py on CPU: two gloo ranks.

With N replicas the benchmark reports every replica's bytes over the
slowest replica's time; this checks the max-over-ranks reduction and the
whole-job formula without a GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = [12.5, 20.0][rank]
    m = bench.max_over_ranks(local_ms)
    gbs = bench.whole_job_gbs(10**9, 4, world, m)
    out.put((rank, m, gbs))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, gbs in res:
        assert m == 20.0  # the slowest replica sets the time on every rank
        # 2 replicas x 4 steps x 1 GB in 20 ms
        assert gbs == pytest.approx(2 * 4 * 1.0 / 0.020)


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_gbs(2 * 10**9, 10, 1, 1000.0) == pytest.approx(20.0)
