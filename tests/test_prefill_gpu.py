"""Sparse prefill attention (plan + attention + combine) on the GPU against
the FP64 oracle, element by element, with the acceptance rule of vLLM PR
60684 (Validation) for the bf16 output and 1e-2 for the fp32 lse."""
import numpy as np
import pytest
import torch

import block_sparse_attention_prefill_gb300 as msa
import oracle
import pins
import workloads
from gpu_cases import check_against_oracle, run_gpu, sample_tokens
from tolerance import assert_acceptance, assert_lse

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(16))
def test_tiny_full_prefill_equals_dense(seed):
    # every visible page is selected: the oracle equals dense causal attention
    w = workloads.make_config("tiny_full_prefill", seed=seed)
    s, e, st = check_against_oracle(w, what="tiny seed %d" % seed)
    assert st == 0


@pytest.mark.parametrize("seed", range(16))
def test_chunked_prefill_32k(seed):
    w = workloads.make_config("chunked_prefill_32k", seed=seed)
    check_against_oracle(w, what="chunked seed %d" % seed)


@pytest.mark.parametrize("seed", range(4))
def test_ragged_batch_8(seed):
    w = workloads.make_config("ragged_batch_8", seed=seed)
    check_against_oracle(w, what="ragged seed %d" % seed)


@pytest.mark.parametrize("hq,hkv", [(16, 1), (12, 4), (8, 8), (4, 1),
                                    (64, 4), (128, 1), (6, 2)])
def test_group_sizes(hq, hkv):
    w = workloads.make_batch("g", [300, 77], [3000, 600], hq, hkv, seed=hq + hkv)
    check_against_oracle(w, what="G=%d" % (hq // hkv))


def test_invalid_entries_are_skipped():
    for seed in (3, 4):
        w = pins.tiny_sparse_workload(seed)
        s, e, st = check_against_oracle(w, what="invalid")
        assert st & msa.STATUS_BAD_PAGE_ID and st & msa.STATUS_BAD_BLOCK


def test_first_token_single_key():
    # position 0 attends to key 0 only: out = bf16(V0 * v_scale)
    w = workloads.make_batch("one", [130], [130], 8, 2, seed=12)
    out, lse, plan, _ = run_gpu(w)
    ro, rl, _ = oracle.attention(w, tokens=[0])
    ref = torch.from_numpy(ro[0]).to(torch.bfloat16).float().numpy()
    got = out[0]
    ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
    assert (np.abs(got - ref) <= ulp).all()
    assert np.abs(lse[0] - rl[0]).max() < 1e-3


def test_block_table_permutation_bitwise():
    w = workloads.make_batch("perm", [200, 90], [5000, 1400], 16, 2, seed=13)
    out, lse, _, _ = run_gpu(w)
    g = torch.Generator().manual_seed(3)
    perm = torch.randperm(w.num_pages, generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(w.num_pages)
    bt2 = torch.where(w.block_table >= 0,
                      inv[w.block_table.long().clamp(min=0)].to(torch.int32),
                      w.block_table)
    w2 = pins._replace(w, kv=w.kv[perm].contiguous(), block_table=bt2)
    out2, lse2, _, _ = run_gpu(w2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_all_padding_gives_zeros():
    w = workloads.make_batch("pad", [40], [3000], 8, 2, seed=14)
    w = pins._replace(w, topk=torch.full_like(w.topk, -1))
    out, lse, plan, _ = run_gpu(w)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_empty_batch():
    w = workloads.make_batch("empty", [0], [500], 8, 2, seed=15)
    out, lse, plan, _ = run_gpu(w)
    assert out.shape == (0, 8, 128)


def test_long_rows_from_empty_cache():
    # page 0 is selected by ~4700 tokens of 8192: many chunks per row
    w = workloads.make_batch("ctx0", [8192], [8192], 16, 1, seed=16)
    toks = sample_tokens(w.T, 96, seed=1)
    check_against_oracle(w, tokens=toks, what="ctx0")


@pytest.mark.parametrize("name", ["long_prefill_150k", "long_prefill_1m"])
def test_full_size_all_tokens(name):
    # the bench's workloads at full size, every token against the oracle
    w = workloads.make_config(name, seed=0)
    s, e, st = check_against_oracle(w, what=name)
    assert st == 0


def test_repeatable_and_stream_ordered():
    w = workloads.make_config("chunked_prefill_32k", seed=5).to("cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1, _ = msa.run_workload(w)
        o2, l2, _ = msa.run_workload(w)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("name", ["chunked_prefill_32k", "long_prefill_1m"])
def test_one_plan_serves_repeated_launches(name):
    # one plan, several prefill launches on one workspace: each (token,
    # head, slot) partial has exactly one writer, so the results are
    # bit-identical launch after launch
    w = workloads.make_config(name, seed=3).to("cuda")
    plan = msa.msa_plan(w.topk, w.cu_q, w.cu_k, w.block_table, w.num_pages,
                        w.Hq, w.total_rows, w.max_seqlen_q, w.max_seqlen_k)
    ws = torch.empty(msa.prefill_workspace_bytes(w.T, w.Hq),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(4):
        out, lse = msa.msa_prefill(w.q, w.kv, w.q_scale, w.k_scale, w.v_scale,
                                   w.softmax_scale, w.block_table, plan,
                                   workspace=ws)
        outs.append((out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert plan.status() == 0
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


@pytest.mark.parametrize("seed", [0, 1])
def test_mixed_decode_and_prefill_batch(seed):
    # decode / speculative-verify requests (1 to 8 tokens at the tail of a
    # long context) and chunked prefills in one plan and one prefill call,
    # decodes first as the serving engine orders them
    w = workloads.make_batch("mixed", [1, 8, 4, 8, 333, 1024],
                             [40000, 65536, 9000, 131072, 5000, 1024],
                             16, 2, seed=40 + seed)
    s, e, st = check_against_oracle(w, what="mixed seed %d" % seed)
    assert st == 0


def test_large_outputs_keep_the_acceptance_rule():
    # outputs near +-19 with exact probabilities (pins.flat_large_v_workload):
    # partials rounded to E4M3 alone would break the rule of vLLM PR 60684
    # (Validation) on a sixth of the elements; the kernel keeps such halves
    # in bf16, so the rule holds here as on the pages' own inputs
    w = pins.flat_large_v_workload(0)
    s, e, st = check_against_oracle(w, what="large |out|")
    assert st == 0
