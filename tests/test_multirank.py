"""bench.py's multi-rank logic on CPU with gloo, world size 2: max-over-ranks
timing, the whole-job weak-scaling rate, and the reference arm's non-zero
ranks exiting without work."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    seconds = [0.25, 0.40][rank]
    slowest = bench.max_over_ranks(seconds, dist)
    rate = bench.whole_job_rate(1_000_000_000, slowest, world)
    dist.barrier()
    if rank == 1:
        # the reference arm: ranks other than 0 leave at once, without work
        bench.reference_arm(None, world, rank, dist)
        results[rank] = (slowest, rate, "left")
    else:
        dist.destroy_process_group()
        results[rank] = (slowest, rate, "done")


def test_two_gloo_ranks():
    world = 2
    port = free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert res[0][0] == res[1][0] == pytest.approx(0.40)
    assert res[0][1] == pytest.approx(2 * 1.0 / 0.40)
    assert res[1][2] == "left" and res[0][2] == "done"
