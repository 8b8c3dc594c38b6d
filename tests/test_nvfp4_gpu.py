"""NVFP4 K/V pages (vLLM PR 60684, Details: with an E4M3 query each NVFP4
code times its block scale is dequantised to E4M3, the K global scale goes
on the scores and the V global scale into the combine).

- The staging kernel (msa_nvfp4_to_e4m3) against the oracle's conversion,
  bit for bit, over every code and every finite block scale.
- msa_prefill_nvfp4 / msa_decode_nvfp4 against the FP64 oracle on the same
  NVFP4 pool, under the acceptance rule of vLLM PR 60684 (Validation).
- The fused path (NVFP4 pages dequantised in shared memory) against
  msa_prefill on the staged E4M3 pool: the same tiles reach the same MMAs,
  so the outputs are identical bit for bit.
"""
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

SLOT = msa.NVFP4_SLOT_BYTES
CODES = 128 * 64


def _random_pool(pages, hkv, seed):
    """Random code bytes; block scales drawn from every finite E4M3 code,
    both signs (0x7F and 0xFF are NaN, not scales)."""
    rng = np.random.default_rng(seed)
    kv4 = rng.integers(0, 256, size=(pages, hkv, 2, SLOT), dtype=np.uint8)
    sc = kv4[..., CODES:]
    sc[(sc & 0x7F) == 0x7F] ^= 0x01
    return torch.from_numpy(kv4)


@pytest.mark.parametrize("pages,hkv,seed", [(1, 1, 0), (37, 3, 1), (300, 2, 2)])
def test_staging_bit_exact(pages, hkv, seed):
    kv4 = _random_pool(pages, hkv, seed)
    got = msa.msa_nvfp4_to_e4m3(kv4.cuda())
    torch.cuda.synchronize()
    want = oracle.nvfp4_to_e4m3(kv4)
    assert np.array_equal(got.view(torch.uint8).cpu().numpy(), want)


def test_staging_covers_every_code_and_scale():
    # one page-head per scale code: every (E2M1 code, scale) pair appears
    scales = [c for c in range(256) if (c & 0x7F) != 0x7F]
    kv4 = np.zeros((len(scales), 1, 2, SLOT), np.uint8)
    pair = np.arange(256, dtype=np.uint8)          # byte = two E2M1 codes
    kv4[:, :, :, :CODES] = np.tile(pair, CODES // 256)
    for i, c in enumerate(scales):
        kv4[i, :, :, CODES:] = c
    got = msa.msa_nvfp4_to_e4m3(torch.from_numpy(kv4).cuda())
    torch.cuda.synchronize()
    want = oracle.nvfp4_to_e4m3(kv4)
    assert np.array_equal(got.view(torch.uint8).cpu().numpy(), want)


@pytest.mark.parametrize("name", ["tiny_full_prefill_nvfp4",
                                  "chunked_prefill_32k_nvfp4",
                                  "ragged_batch_8_nvfp4"])
def test_prefill_nvfp4_matches_oracle(name):
    w = workloads.make_config(name, seed=3)
    s, e, st = check_against_oracle(w, what=name)
    assert st == 0


@pytest.mark.parametrize("hq,hkv", [(16, 1), (12, 4), (6, 2), (128, 1)])
def test_prefill_nvfp4_group_sizes(hq, hkv):
    # G = 16, 3, 3, 128: Q rows by TMA and by the converter warps' gather
    w = workloads.make_batch("g4", [300, 77], [3000, 600], hq, hkv,
                             seed=hq + hkv, kv_format="nvfp4")
    check_against_oracle(w, what="nvfp4 G=%d" % (hq // hkv))


@pytest.mark.parametrize("name", ["chunked_prefill_32k_nvfp4",
                                  "ragged_batch_8_nvfp4"])
def test_fused_equals_staged(name):
    w = workloads.make_config(name, seed=5).to("cuda")
    out4, lse4, plan = msa.run_workload(w)
    kv8 = msa.msa_nvfp4_to_e4m3(w.kv4)
    out8, lse8 = msa.msa_prefill(w.q, kv8, w.q_scale, w.k_scale, w.v_scale,
                                 w.softmax_scale, w.block_table, plan)
    torch.cuda.synchronize()
    assert torch.equal(out4, out8) and torch.equal(lse4, lse8)


@pytest.mark.parametrize("name", ["long_prefill_1m_nvfp4",
                                  "long_prefill_150k_nvfp4"])
def test_full_size_all_tokens(name):
    # the bench's NVFP4 workloads at full size, every token against the oracle
    w = workloads.make_config(name, seed=0)
    s, e, st = check_against_oracle(w, what=name)
    assert st == 0


def test_decode_nvfp4_matches_oracle():
    w = workloads.make_config("decode_16x8_nvfp4", seed=1)
    wd = w.to("cuda")
    n = w.q_lens[0]
    seq = torch.tensor(w.seq_lens, dtype=torch.int32, device="cuda")
    out, lse, plan = msa.msa_decode_nvfp4(wd.q, wd.kv4, w.q_scale, w.k_scale,
                                          w.v_scale, w.softmax_scale, wd.topk,
                                          wd.block_table, seq, n,
                                          w.max_seqlen_k)
    torch.cuda.synchronize()
    assert plan.status() == 0
    ro, rl, _ = oracle.attention(w)
    assert_acceptance(out.float().cpu().numpy(), ro, "decode nvfp4")
    assert_lse(lse.cpu().numpy(), rl, "decode nvfp4")
    # the same kernels through the prefill entry points: identical bits
    o2, l2, _ = msa.run_workload(wd)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_nvfp4_invalid_entries_are_skipped():
    # planted bad ids, repeats, future pages and a bad block-table entry, as
    # in the E4M3 test, over an NVFP4 pool
    w = workloads.make_batch("tiny_sparse4", [5, 3, 4], [2400, 300, 130], 4, 2,
                             seed=3, kv_format="nvfp4")
    tk = w.topk.clone()
    tk[0, 0, 5] = 10**6
    tk[1, 1, 3] = -7
    tk[2, 0, 7] = tk[2, 0, 1]
    tk[8, 0, 3] = 1
    bt = w.block_table.clone()
    bt[0, 3] = -1
    w = pins._replace(w, topk=tk, block_table=bt)
    s, e, st = check_against_oracle(w, what="nvfp4 invalid")
    assert st & msa.STATUS_BAD_PAGE_ID and st & msa.STATUS_BAD_BLOCK


def test_nvfp4_graph_replay_matches_eager():
    w = workloads.make_config("chunked_prefill_32k_nvfp4", seed=7).to("cuda")
    ws_plan = torch.empty(msa.plan_workspace_bytes(
        w.B, w.T, w.Hq, w.Hkv, w.total_rows, w.max_seqlen_q),
        dtype=torch.uint8, device="cuda")
    ws_pre = torch.empty(msa.prefill_workspace_bytes(w.T, w.Hq),
                         dtype=torch.uint8, device="cuda")
    out = torch.empty((w.T, w.Hq, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.T, w.Hq), dtype=torch.float32, device="cuda")

    def step():
        plan = msa.msa_plan(w.topk, w.cu_q, w.cu_k, w.block_table, w.num_pages,
                            w.Hq, w.total_rows, w.max_seqlen_q, w.max_seqlen_k,
                            workspace=ws_plan)
        msa.msa_prefill_nvfp4(w.q, w.kv4, w.q_scale, w.k_scale, w.v_scale,
                              w.softmax_scale, w.block_table, plan,
                              workspace=ws_pre, out=out, lse=lse)
        return plan

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan = step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert plan.status() == 0
    ref = [out.clone(), lse.clone()]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])


def test_nvfp4_binding_rejects_wrong_pool_shape():
    w = workloads.make_config("tiny_full_prefill_nvfp4", seed=0).to("cuda")
    plan = msa.msa_plan(w.topk, w.cu_q, w.cu_k, w.block_table, w.num_pages,
                        w.Hq, w.total_rows, w.max_seqlen_q, w.max_seqlen_k)
    with pytest.raises(msa.MsaError):
        msa.msa_prefill_nvfp4(w.q, w.kv4.view(w.num_pages, w.Hkv, -1),
                              w.q_scale, w.k_scale, w.v_scale,
                              w.softmax_scale, w.block_table, plan)
