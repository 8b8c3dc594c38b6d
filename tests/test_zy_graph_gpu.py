"""CUDA-graph capture of the hot calls.

msa_plan + msa_prefill, and msa_decode, are captured once with
preallocated workspaces and outputs, then replayed. Every kernel is
deterministic, so each replay must reproduce the eager result bit for bit.
The plan's kernels, the attention kernel and the combine are programmatic
dependent launches, which a capture keeps as graph edges.
"""
import pytest
import torch

import block_sparse_attention_prefill_gb300 as msa
import workloads

pytestmark = pytest.mark.gpu


def _capture_and_replay(step, outputs, replays=3):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan = step()  # eager: also the one-time launch attributes
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert plan.status() == 0
    ref = [o.clone() for o in outputs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(replays):
        for o in outputs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for o, r in zip(outputs, ref):
            assert torch.equal(o, r)


@pytest.mark.parametrize("name", ["chunked_prefill_32k", "ragged_batch_8"])
def test_prefill_graph_replay_matches_eager(name):
    w = workloads.make_config(name, seed=7).to("cuda")
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
        msa.msa_prefill(w.q, w.kv, w.q_scale, w.k_scale, w.v_scale,
                        w.softmax_scale, w.block_table, plan, workspace=ws_pre,
                        out=out, lse=lse)
        return plan

    _capture_and_replay(step, [out, lse])


def test_decode_graph_replay_matches_eager():
    w = workloads.make_config("decode_16x8", seed=3).to("cuda")
    n = int(w.q_lens[0])
    seq_lens = torch.tensor(w.seq_lens, dtype=torch.int32, device="cuda")
    ws = torch.empty(msa.decode_workspace_bytes(w.B, n, w.Hq, w.Hkv,
                                                w.max_seqlen_k),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((w.T, w.Hq, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.T, w.Hq), dtype=torch.float32, device="cuda")

    def step():
        _, _, plan = msa.msa_decode(w.q, w.kv, w.q_scale, w.k_scale, w.v_scale,
                                    w.softmax_scale, w.topk, w.block_table,
                                    seq_lens, n, w.max_seqlen_k, workspace=ws,
                                    out=out, lse=lse)
        return plan

    _capture_and_replay(step, [out, lse])
