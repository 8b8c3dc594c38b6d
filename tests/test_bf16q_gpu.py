"""The BF16-query mode (BF16 Q over the E4M3 pool, K/V widened to bf16,
bf16 MMAs) on the GPU against the FP64 oracle, element by element, with the
acceptance rule of vLLM PR 60684 (Validation) for the bf16 output and 1e-2
for the fp32 lse; the plan and the combine are those of the E4M3 query."""
import numpy as np
import pytest
import torch

import block_sparse_attention_prefill_gb300 as msa
import pins
import workloads
from gpu_cases import check_against_oracle, run_gpu, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(4))
def test_tiny_full_prefill_equals_dense(seed):
    w = workloads.make_config("tiny_full_prefill_bf16q", seed=seed)
    s, e, st = check_against_oracle(w, what="bf16q tiny seed %d" % seed)
    assert st == 0


@pytest.mark.parametrize("seed", range(16))
def test_chunked_prefill_32k(seed):
    w = workloads.make_config("chunked_prefill_32k_bf16q", seed=seed)
    check_against_oracle(w, what="bf16q chunked seed %d" % seed)


def test_ragged_batch_8():
    w = workloads.make_config("ragged_batch_8_bf16q", seed=0)
    check_against_oracle(w, what="bf16q ragged")


@pytest.mark.parametrize("hq,hkv", [(16, 1), (12, 4), (8, 8), (4, 1),
                                    (64, 4), (128, 1), (6, 2)])
def test_group_sizes(hq, hkv):
    w = workloads.with_bf16_query(
        workloads.make_batch("g", [300, 77], [3000, 600], hq, hkv, seed=hq + hkv),
        seed=hq)
    check_against_oracle(w, what="bf16q G=%d" % (hq // hkv))


def test_invalid_entries_are_skipped():
    for seed in (3, 4):
        w = workloads.with_bf16_query(pins.tiny_sparse_workload(seed), seed=seed)
        s, e, st = check_against_oracle(w, what="bf16q invalid")
        assert st & msa.STATUS_BAD_PAGE_ID and st & msa.STATUS_BAD_BLOCK


def test_widened_e4m3_query_with_its_scale():
    # the E4M3 query widened to bf16 (exact) with its own q_scale: the
    # oracle of this input is the E4M3-query oracle, bit for bit
    w = workloads.make_config("chunked_prefill_32k", seed=7)
    q16 = w.q.view(torch.float8_e4m3fn).to(torch.bfloat16)
    wb = pins._replace(w, q=None, q16=q16)
    check_against_oracle(wb, tokens=sample_tokens(w.T, 128, seed=2),
                         what="bf16q widened")


@pytest.mark.parametrize("seed", range(2))
def test_mixed_decode_and_prefill_batch(seed):
    # decode / speculative-verify requests and chunked prefills in one plan
    # and one call, decodes first
    w = workloads.with_bf16_query(
        workloads.make_batch("mixed", [1, 8, 4, 8, 333, 1024],
                             [40000, 65536, 9000, 131072, 5000, 1024], 16, 2,
                             seed=40 + seed), seed=seed)
    s, e, st = check_against_oracle(w, what="bf16q mixed seed %d" % seed)
    assert st == 0


def test_large_outputs_keep_the_acceptance_rule():
    # outputs near +-19 (flat softmax, V codes near +-300): the partial
    # halves above the E4M3 limit go to the bf16 overflow rows here too
    w = workloads.with_bf16_query(pins.flat_large_v_workload(0))
    s, e, st = check_against_oracle(w, what="bf16q large |out|")
    assert st == 0


def test_head_shards_equal_the_whole():
    # the plan of each KV-head shard (msa_plan_heads) with the shard's own
    # BF16 query and pool reproduces the unsharded result bit for bit
    w = workloads.make_config("chunked_prefill_32k_bf16q", seed=3).to("cuda")
    out, lse, _ = msa.run_workload(w)
    G = w.G
    for h0 in range(w.Hkv):
        plan = msa.msa_plan(w.topk, w.cu_q, w.cu_k, w.block_table, w.num_pages, G,
                            w.total_rows, w.max_seqlen_q, w.max_seqlen_k,
                            h_begin=h0, h_count=1)
        q = w.q16[:, h0 * G:(h0 + 1) * G].contiguous()
        kv = w.kv[:, h0:h0 + 1].contiguous()
        o, l = msa.msa_prefill_bf16q(q, kv, w.q_scale, w.k_scale, w.v_scale,
                                     w.softmax_scale, w.block_table, plan)
        torch.cuda.synchronize()
        assert torch.equal(o, out[:, h0 * G:(h0 + 1) * G])
        assert torch.equal(l, lse[:, h0 * G:(h0 + 1) * G])


def test_all_padding_gives_zeros():
    w = workloads.with_bf16_query(workloads.make_batch("pad", [40], [3000], 8, 2, seed=14))
    w = pins._replace(w, topk=torch.full_like(w.topk, -1))
    out, lse, plan, _ = run_gpu(w)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_first_token_single_key():
    # position 0 attends to key 0 only: out = bf16(V0 * v_scale)
    w = workloads.with_bf16_query(workloads.make_batch("one", [130], [130], 8, 2, seed=12))
    out, lse, plan, _ = run_gpu(w)
    import oracle
    ro, rl, _ = oracle.attention(w, tokens=[0])
    ref = torch.from_numpy(ro[0]).to(torch.bfloat16).float().numpy()
    assert (np.abs(out[0] - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30).all()
    assert np.abs(lse[0] - rl[0]).max() < 1e-3


def test_halves_equal_the_one_call():
    w = workloads.make_config("ragged_batch_8_bf16q", seed=1).to("cuda")
    out1, lse1, plan = msa.run_workload(w)
    ws = torch.empty(msa.prefill_workspace_bytes(w.T, w.Hq), dtype=torch.uint8,
                     device="cuda")
    msa.msa_prefill_attention_bf16q(w.q16, w.kv, w.q_scale, w.k_scale, w.v_scale,
                                    w.softmax_scale, w.block_table, plan, ws)
    out2 = torch.empty_like(out1)
    lse2 = torch.empty_like(lse1)
    msa.msa_prefill_combine(plan, ws, out2, lse2)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


@pytest.mark.parametrize("name", ["long_prefill_150k_bf16q", "long_prefill_1m_bf16q"])
def test_full_size(name):
    w = workloads.make_config(name, seed=0)
    toks = None if name.endswith("1m_bf16q") else sample_tokens(w.T, 512, seed=3)
    s, e, st = check_against_oracle(w, tokens=toks, what=name)
    assert st == 0


def test_short_wait_limit_expires_and_the_next_call_is_clean():
    lib = msa.load()
    w = workloads.make_config("chunked_prefill_32k_bf16q", seed=2).to("cuda")
    ref_o, ref_l, plan = msa.run_workload(w)
    torch.cuda.synchronize()
    assert plan.status() == 0
    try:
        # 1 ns: every wait for an MMA that has not completed when the clock
        # next moves runs out
        assert lib.msa_test_set_wait_limit_ns(1) == 0
        _, _, plan = msa.run_workload(w)
        torch.cuda.synchronize()
        assert plan.status() & msa.STATUS_TIMEOUT
    finally:
        lib.msa_test_set_wait_limit_ns(0)
    o, l, plan = msa.run_workload(w)
    torch.cuda.synchronize()
    assert plan.status() == 0
    assert torch.equal(o, ref_o) and torch.equal(l, ref_l)
