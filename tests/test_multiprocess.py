"""The multi-GPU bookkeeping of bench.py on CPU: two gloo ranks.

Rows are independent, so ranks never exchange data; the only collective is
the max over ranks of the timed region, and the whole-job rate counts every
rank's rows.  Each rank reports a different time; both must see the larger,
and the rate must be world * rows / that time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank          # rank 1 is the slower one
    got = bench.max_over_ranks(ms, world, "cpu")
    out[rank] = (got, bench.whole_job_rate(world, 256, got))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == res[1][1] == pytest.approx(2 * 256 / 0.015)


def test_single_rank_needs_no_collective():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_rate(1, 256, 2.0) == pytest.approx(128000.0)
