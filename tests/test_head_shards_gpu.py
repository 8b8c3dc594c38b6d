"""Head sharding as a parameter (KV heads [h_begin, h_begin + h_count) of a
shared top-k tensor, the rank's own Q, pool and output): under tensor
parallelism a rank holds num_attention_heads // tp_size query heads and the
KV heads of its cache (vLLM docs, sparse_attention_msa,
MiniMaxM3SparseMSAMetadataBuilder), and the heads shard with no exchange.
Every shard must reproduce its heads of the unsharded call bit for bit:
the same work items, MMAs and merges per head."""
import pytest
import torch

import block_sparse_attention_prefill_gb300 as msa
import workloads

pytestmark = pytest.mark.gpu


def _prefill(w, q, kv, topk, Hq, h_begin=None, h_count=None):
    plan = msa.msa_plan(topk, w.cu_q, w.cu_k, w.block_table, w.num_pages, Hq,
                        w.total_rows, w.max_seqlen_q, w.max_seqlen_k,
                        h_begin=h_begin, h_count=h_count)
    out, lse = msa.msa_prefill(q, kv, w.q_scale, w.k_scale, w.v_scale,
                               w.softmax_scale, w.block_table, plan)
    torch.cuda.synchronize()
    assert plan.status() == 0
    return out, lse, plan


@pytest.mark.parametrize("name,shards", [
    ("chunked_prefill_32k", [(0, 1), (1, 1)]),
    ("ragged_batch_8", [(0, 1), (1, 1)]),
])
def test_head_shards_match_the_unsharded_call(name, shards):
    w = workloads.make_config(name, seed=4).to("cuda")
    G = w.Hq // w.Hkv
    out, lse, _ = _prefill(w, w.q, w.kv, w.topk, w.Hq)
    for h0, hn in shards:
        qs = w.q[:, h0 * G:(h0 + hn) * G].contiguous()
        kvs = w.kv[:, h0:h0 + hn].contiguous()
        o, l, plan = _prefill(w, qs, kvs, w.topk, hn * G, h_begin=h0, h_count=hn)
        assert torch.equal(o, out[:, h0 * G:(h0 + hn) * G])
        assert torch.equal(l, lse[:, h0 * G:(h0 + hn) * G])


def test_four_shards_of_a_wider_batch():
    # Hkv 4, Hq 16 (G 4): four one-head shards and one two-head shard
    w = workloads.make_batch("shards", [300, 57, 1024], [3000, 57, 9000], 16, 4,
                             seed=21).to("cuda")
    G = w.Hq // w.Hkv
    out, lse, full = _prefill(w, w.q, w.kv, w.topk, w.Hq)
    nnz_full, _ = full.counters()
    nnz = 0
    for h0, hn in [(0, 1), (1, 1), (2, 1), (3, 1), (1, 2)]:
        qs = w.q[:, h0 * G:(h0 + hn) * G].contiguous()
        kvs = w.kv[:, h0:h0 + hn].contiguous()
        o, l, plan = _prefill(w, qs, kvs, w.topk, hn * G, h_begin=h0, h_count=hn)
        assert torch.equal(o, out[:, h0 * G:(h0 + hn) * G])
        assert torch.equal(l, lse[:, h0 * G:(h0 + hn) * G])
        if hn == 1:
            nnz += plan.counters()[0]
    # the one-head shards' CSRs partition the unsharded one
    assert nnz == nnz_full
