"""The bounded-wait expiry path of the attention kernel, on the GPU, without
faulting or hanging anything: a test-only hook shortens the pipeline waits'
wall-time limit below a page load, so a wait runs out on a real workload.
The call must still return, the plan's status word must carry
MSA_STATUS_TIMEOUT, and the next call on the same workspaces, with the
default limit back, must give exactly the clean result."""
import pytest
import torch

import block_sparse_attention_prefill_gb300 as msa
import workloads

pytestmark = pytest.mark.gpu


def _step(w, ws_plan, ws_pre, out, lse):
    plan = msa.msa_plan(w.topk, w.cu_q, w.cu_k, w.block_table, w.num_pages,
                        w.Hq, w.total_rows, w.max_seqlen_q, w.max_seqlen_k,
                        workspace=ws_plan)
    msa.msa_prefill(w.q, w.kv, w.q_scale, w.k_scale, w.v_scale,
                    w.softmax_scale, w.block_table, plan, workspace=ws_pre,
                    out=out, lse=lse)
    torch.cuda.synchronize()
    return plan


def test_short_wait_limit_expires_and_the_next_call_is_clean():
    lib = msa.load()
    w = workloads.make_config("chunked_prefill_32k", seed=2).to("cuda")
    ws_plan = torch.empty(msa.plan_workspace_bytes(
        w.B, w.T, w.Hq, w.Hkv, w.total_rows, w.max_seqlen_q),
        dtype=torch.uint8, device="cuda")
    ws_pre = torch.empty(msa.prefill_workspace_bytes(w.T, w.Hq),
                         dtype=torch.uint8, device="cuda")
    out = torch.empty((w.T, w.Hq, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.T, w.Hq), dtype=torch.float32, device="cuda")
    plan = _step(w, ws_plan, ws_pre, out, lse)
    assert plan.status() == 0
    ref_o, ref_l = out.clone(), lse.clone()
    try:
        # 300 ns: far below the latency of a K|V page load, so the first
        # wait on one runs out
        assert lib.msa_test_set_wait_limit_ns(300) == 0
        plan = _step(w, ws_plan, ws_pre, out, lse)
        assert plan.status() & msa.STATUS_TIMEOUT
    finally:
        lib.msa_test_set_wait_limit_ns(0)
    # the context is usable, and the workspaces carry nothing over
    plan = _step(w, ws_plan, ws_pre, out, lse)
    assert plan.status() == 0
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
