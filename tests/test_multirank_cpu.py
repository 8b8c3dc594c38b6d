"""The multi-GPU host logic of bench.py with two gloo ranks on CPU: every
rank gets its own batch (its own seed), timings are reduced by max and work
by sum, and the whole-job rate is the summed work over the slowest rank.
No data is exchanged between ranks (each request / KV head is independent),
so this is all the N > 1 path adds."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port,
                            rank=rank, world_size=world)
    try:
        seed = bench.rank_seed(7, rank)
        times = bench.reduce_over_ranks([1.0 + rank, 5.0 - rank], world, "cpu",
                                        "max")
        (pairs,) = bench.reduce_over_ranks([1000.0 * (rank + 1)], world, "cpu",
                                           "sum")
        dist.barrier()
        out[rank] = (seed, times, pairs, bench.job_tflops(pairs, times[0]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world,
                       start_method="spawn", join=True)
    r0, r1 = out[0], out[1]
    assert r0[0] != r1[0]                       # independent batches
    assert r0[1] == r1[1] == [2.0, 5.0]         # max over ranks
    assert r0[2] == r1[2] == 3000.0             # work summed
    assert r0[3] == pytest.approx(4 * 128 * 3000.0 / 2e-3 / 1e12)
