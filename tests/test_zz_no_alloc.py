"""msa_decode_noalloc: decode for callers that cannot allocate device
memory (they pass only raw device pointers and have no allocator to call).
It keeps its scratch in one fixed device array inside the library, so these
checks compare it with msa_decode, which uses a caller-owned workspace, on
two calls in a row (the second call finds the first call's data in the
shared array), and check that a batch too large for the array is refused.
This file is collected last so a stop-at-first-failure run has already run
every other test."""
import ctypes

import pytest
import torch

import block_sparse_attention_prefill_gb300 as msa
import workloads
from tolerance import assert_acceptance, assert_lse

pytestmark = pytest.mark.gpu


def _batch(seed, B, n):
    sl = workloads.decode_lengths(seed, B, 2000, 40000)
    return workloads.make_batch("noalloc", [n] * B, sl, 16, 2, seed=seed).to("cuda")


def _both(w, n):
    seq = torch.tensor(w.seq_lens, dtype=torch.int32, device="cuda")
    ref_o, ref_l, _ = msa.msa_decode(w.q, w.kv, w.q_scale, w.k_scale, w.v_scale,
                                     w.softmax_scale, w.topk, w.block_table,
                                     seq, n, w.max_seqlen_k)
    out = torch.full_like(ref_o, float("nan"))
    lse = torch.full_like(ref_l, float("nan"))
    msa.msa_decode_noalloc(w.q, w.kv, w.q_scale, w.k_scale, w.v_scale,
                           w.softmax_scale, w.topk, w.block_table, seq, n,
                           w.max_seqlen_k, out, lse)
    torch.cuda.synchronize()
    return ref_o, ref_l, out, lse


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    # the two calls run the same deterministic kernels on the same inputs, so
    # the results agree bit for bit (and so within any tolerance)
    for seed, B, n in ((0, 12, 8), (1, 5, 3)):
        w = _batch(seed, B, n)
        ref_o, ref_l, out, lse = _both(w, n)
        assert torch.equal(out, ref_o), "noalloc seed %d: out differs" % seed
        assert torch.equal(lse, ref_l), "noalloc seed %d: lse differs" % seed
        assert_acceptance(out.float().cpu().numpy(), ref_o.float().cpu().numpy(),
                          "noalloc seed %d" % seed)
        assert_lse(lse.cpu().numpy(), ref_l.cpu().numpy(), "noalloc seed %d" % seed)


def test_noalloc_refuses_a_batch_beyond_its_scratch():
    lib = msa.load()
    need = msa.decode_workspace_bytes(64, 8, 16, 2, 131072)
    assert need > 16 << 20
    fake = ctypes.c_void_p(4096)  # never dereferenced: refused on the host
    rc = lib.msa_decode_noalloc(fake, fake, 100, 1.0, 1.0, 1.0, 0.1, fake, fake,
                                1024, fake, 64, 8, 16, 2, 131072, fake, None,
                                None)
    assert rc == 7 and "scratch" in msa.status_string(rc)
