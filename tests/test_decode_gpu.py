"""Decode / speculative verify (8 query tokens per request at the tail of
32K-131K contexts) against the FP64 oracle, and bit-identical to planning
the same batch as a prefill."""
import numpy as np
import pytest
import torch

import block_sparse_attention_prefill_gb300 as msa
import oracle
import workloads
from tolerance import assert_acceptance, assert_lse

pytestmark = pytest.mark.gpu


def run_decode(w):
    wd = w.to("cuda")
    n = w.q_lens[0]
    seq = torch.tensor(w.seq_lens, dtype=torch.int32, device="cuda")
    out, lse, plan = msa.msa_decode(wd.q, wd.kv, w.q_scale, w.k_scale,
                                    w.v_scale, w.softmax_scale, wd.topk,
                                    wd.block_table, seq, n, w.max_seqlen_k)
    torch.cuda.synchronize()
    return out, lse, plan, wd


@pytest.mark.parametrize("name", ["decode_16x8", "decode_64x8"])
def test_decode_matches_oracle(name):
    w = workloads.make_config(name, seed=0, kv_device="cuda")
    out, lse, plan, wd = run_decode(w)
    assert plan.status() == 0
    ro, rl, _ = oracle.attention(w.to("cpu"))
    assert_acceptance(out.float().cpu().numpy(), ro, name)
    assert_lse(lse.cpu().numpy(), rl, name)
    # same kernels through the prefill entry points: identical bits
    o2, l2, _ = msa.run_workload(wd)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("n", [1, 2, 4])
def test_decode_short_drafts(n):
    sl = workloads.decode_lengths(1, 12, 300, 9000)
    w = workloads.make_batch("dec", [n] * 12, sl, 16, 2, seed=n)
    out, lse, plan, _ = run_decode(w)
    ro, rl, _ = oracle.attention(w)
    assert_acceptance(out.float().cpu().numpy(), ro, "n=%d" % n)
    assert_lse(lse.cpu().numpy(), rl, "n=%d" % n)
