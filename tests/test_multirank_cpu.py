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


def _shard_main(rank, world, port, out):
    # KV-head sharding on two gloo ranks: each rank attends its own KV head
    # (the topk slice [:, h, :], its query heads, its pool heads) with the
    # FP64 oracle; nothing is exchanged inside the path.  The gather here is
    # only the check: the shards put together equal the unsharded result.
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import block_sparse_attention_prefill_gb300 as msa
    import oracle
    import workloads
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port,
                            rank=rank, world_size=world)
    try:
        w = workloads.make_batch("tp", [40, 9], [600, 300], 8, 2, seed=13)
        G = w.Hq // w.Hkv
        h0, hn = msa.head_shard(w.Hkv, world, rank)
        shard = workloads.Workload(
            w.name, list(w.q_lens), list(w.seq_lens), hn * G, hn,
            q=w.q[:, h0 * G:(h0 + hn) * G].contiguous(),
            kv=w.kv[:, h0:h0 + hn].contiguous(),
            topk=w.topk[:, h0:h0 + hn].contiguous(), block_table=w.block_table,
            cu_q=w.cu_q, cu_k=w.cu_k, q_scale=w.q_scale, k_scale=w.k_scale,
            v_scale=w.v_scale, softmax_scale=w.softmax_scale)
        o, l, _ = oracle.attention(shard, nthreads=1)
        parts = [None] * world
        dist.all_gather_object(parts, (h0, hn, o, l))
        if rank == 0:
            full_o, full_l, _ = oracle.attention(w, nthreads=1)
            got_o = np.concatenate([p[2] for p in sorted(parts, key=lambda p: p[0])], axis=1)
            got_l = np.concatenate([p[3] for p in sorted(parts, key=lambda p: p[0])], axis=1)
            out["ranges"] = [(p[0], p[1]) for p in parts]
            out["equal"] = bool(np.array_equal(got_o, full_o) and np.array_equal(got_l, full_l))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_kv_heads():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_shard_main, args=(world, port, out), nprocs=world,
                       start_method="spawn", join=True)
    assert sorted(out["ranges"]) == [(0, 1), (1, 1)]
    assert out["equal"]


def test_head_shard_ranges():
    import sys
    sys.path.insert(0, ROOT)
    import block_sparse_attention_prefill_gb300 as msa
    assert [msa.head_shard(8, 4, r) for r in range(4)] == [(0, 2), (2, 2), (4, 2), (6, 2)]
    assert msa.head_shard(2, 1, 0) == (0, 2)
    with pytest.raises(msa.MsaError):
        msa.head_shard(6, 4, 0)
