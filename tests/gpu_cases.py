"""Shared helpers of the GPU parity tests: run the CUDA library on a seeded
workload and compare it with the FP64 oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import block_sparse_attention_prefill_gb300 as msa
import oracle
import workloads
from tolerance import assert_acceptance, assert_lse


def run_gpu(w, device="cuda"):
    """Plan + prefill through the C ABI; returns host copies and the plan."""
    wd = w.to(device)
    out, lse, plan = msa.run_workload(wd)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), plan, wd


def check_against_oracle(w, tokens=None, what=""):
    """Element-wise comparison on all tokens (or the listed sample)."""
    out, lse, plan, _ = run_gpu(w)
    st = plan.status()
    ro, rl, _ = oracle.attention(w, tokens=tokens)
    if tokens is not None:
        out = out[np.asarray(tokens)]
        lse = lse[np.asarray(tokens)]
    s = assert_acceptance(out, ro, what)
    e = assert_lse(lse, rl, what)
    return s, e, st


def sample_tokens(T, n=64, seed=0):
    """Evenly spread tokens plus both ends and a few random ones."""
    rng = np.random.default_rng(seed)
    base = np.linspace(0, T - 1, num=min(n, T)).astype(np.int64)
    extra = rng.integers(0, T, size=min(16, T))
    return np.unique(np.concatenate([base, extra, [0, T - 1]]))
