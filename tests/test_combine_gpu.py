"""msa_combine against the FP64 oracle combine: the fp32 path (given fp32
partials) within 1e-2 max abs, bf16 output within bf16 rounding."""
import numpy as np
import pytest
import torch

import block_sparse_attention_prefill_gb300 as msa
import oracle
from tolerance import assert_acceptance, assert_lse

pytestmark = pytest.mark.gpu


def partials(rows, S, seed, empty_frac=0.3, scale=3.0):
    g = torch.Generator().manual_seed(seed)
    po = torch.randn(rows, S, 128, generator=g, dtype=torch.float64)
    pl = torch.randn(rows, S, generator=g, dtype=torch.float64) * scale
    drop = torch.rand(rows, S, generator=g) < empty_frac
    pl[drop] = -np.inf
    pl[: max(1, rows // 50)] = -np.inf            # a few fully empty rows
    return po, pl


@pytest.mark.parametrize("S", [1, 2, 16, 33, 64])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_combine(S, dtype):
    rows = 3001
    po, pl = partials(rows, S, seed=S)
    po_dev = po.to(dtype)
    out, lse = msa.msa_combine(po_dev.cuda(), pl.float().cuda())
    torch.cuda.synchronize()
    ro, rl = oracle.combine(po_dev.double().numpy(), pl.float().double().numpy())
    assert_lse(lse.cpu().numpy(), rl, "combine lse")
    got = out.float().cpu().numpy()
    # fp32 path: error before bf16 rounding is tiny; allow one bf16 ulp
    tol = np.abs(ro) * 2.0 ** -8 + 1e-2
    assert (np.abs(got - ro) <= tol).all()
    empty = np.isneginf(rl)
    assert (got[empty] == 0).all()


def test_combine_large_lse_spread():
    po, pl = partials(512, 16, seed=99, scale=200.0)
    out, lse = msa.msa_combine(po.float().cuda(), pl.float().cuda())
    ro, rl = oracle.combine(po.float().double().numpy(),
                            pl.float().double().numpy())
    assert_lse(lse.cpu().numpy(), rl, "spread lse")
    assert np.isfinite(out.float().cpu().numpy()).all()
