"""Checks that pin the FP64 oracle to facts outside itself.

Each ``check_*`` takes an oracle library handle (the real one, or a copy with
a planted mistake) and raises AssertionError when the oracle disagrees with:
a library routine that computes the same thing in a special case
(torch's scaled_dot_product_attention in float64, torch's E4M3 cast), a
numpy brute force written a different way, a closed form, an invariance the
definition implies, or a plain Python inversion of the page lists.

The attention being pinned is the one defined by vLLM PR 60684 (section
Performance: top-16 of 128-token pages, queries at the tail of the sequence)
and the MSA implementation page of the vLLM docs
(MiniMaxM3SparseMSAImpl.forward: causal=True, page_table=block_table,
seqused_k=seq_lens).
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

import oracle
import workloads
from oracle import oracle as orc

D = 128
PAGE = 128


def _dec_torch(codes) -> np.ndarray:
    t = torch.as_tensor(np.ascontiguousarray(np.asarray(codes, np.uint8)))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _replace(w, **kw):
    d = dict(q=w.q, kv=w.kv, topk=w.topk, block_table=w.block_table,
             cu_q=w.cu_q, cu_k=w.cu_k, kv4=getattr(w, "kv4", None),
             q16=getattr(w, "q16", None))
    d.update(kw)
    return workloads.Workload(w.name, list(w.q_lens), list(w.seq_lens), w.Hq,
                              w.Hkv, q_scale=w.q_scale, k_scale=w.k_scale,
                              v_scale=w.v_scale,
                              softmax_scale=w.softmax_scale, **d)


def _sdpa_reference(w):
    """Dense attention via torch SDPA in float64, valid when every visible
    page of every token is selected (then the sparse key set equals the
    causal prefix)."""
    if w.q16 is not None:
        q = w.q16.to(torch.float64) * w.q_scale
    else:
        q = torch.from_numpy(_dec_torch(w.q.numpy())) * w.q_scale
    kvf = torch.from_numpy(_dec_torch(w.kv.numpy()))
    G = w.G
    outs = []
    for b in range(w.B):
        ql, sl = w.q_lens[b], w.seq_lens[b]
        npg = (sl + PAGE - 1) // PAGE
        phys = w.block_table[b, :npg].long()
        pages = kvf[phys]                      # [npg, Hkv, 128, 256]
        k = pages[..., :D].permute(1, 0, 2, 3).reshape(w.Hkv, npg * PAGE, D)
        v = pages[..., D:].permute(1, 0, 2, 3).reshape(w.Hkv, npg * PAGE, D)
        k = k[:, :sl] * w.k_scale
        v = v[:, :sl] * w.v_scale
        k = k.repeat_interleave(G, dim=0)
        v = v.repeat_interleave(G, dim=0)
        qb = q[int(w.cu_q[b]):int(w.cu_q[b + 1])].permute(1, 0, 2)
        if ql == sl:
            o = torch.nn.functional.scaled_dot_product_attention(
                qb, k, v, is_causal=True, scale=w.softmax_scale)
        else:
            pos = torch.arange(sl - ql, sl)[:, None]
            allowed = torch.arange(sl)[None, :] <= pos
            o = torch.nn.functional.scaled_dot_product_attention(
                qb, k, v, attn_mask=allowed, scale=w.softmax_scale)
        outs.append(o.permute(1, 0, 2))
    return torch.cat(outs, 0).numpy()


def small_dense_workloads():
    """Cases where top-16 covers every visible page (<= 16 pages)."""
    return [
        workloads.make_config("tiny_full_prefill", seed=0),
        workloads.make_batch("chunk_tail", [200], [1500], 8, 2, seed=1),
        workloads.make_batch("two_req", [130, 64], [600, 2048], 8, 1, seed=2),
    ]


def tiny_sparse_workload(seed=3, corrupt=True):
    """A tiny ragged batch with more than 16 visible pages for some tokens,
    plus (optionally) planted invalid entries: ids past the request's pages,
    ids below -1, repeats, future pages, a bad block-table entry."""
    w = workloads.make_batch("tiny_sparse", [5, 3, 4], [2400, 300, 130], 4, 2,
                             seed=seed)
    if corrupt:
        tk = w.topk.clone()
        tk[0, 0, 5] = 10**6           # past the request's pages
        tk[1, 1, 3] = -7              # below -1
        tk[2, 0, 7] = tk[2, 0, 1]     # repeat
        tk[8, 0, 3] = 1               # after the own page (pos 126, page 0)
        tk[9, 1, 2] = 0
        tk[9, 1, 5] = 0               # repeat of a valid id
        tk[3, 0, 9] = 3
        tk[4, 1, 10] = 3
        bt = w.block_table.clone()
        bt[0, 3] = -1                 # request 0, page 3: bad physical page
        w = _replace(w, topk=tk, block_table=bt)
    return w


def flat_large_v_workload(seed=0):
    """Outputs of large magnitude with exact probabilities: every K row is
    the same (so each row's scores are all equal, the softmax is flat and
    the probabilities 2^8 are exact in E4M3), and V codes have magnitudes
    around 300 with a fixed sign per column, so every page's partial and the
    output sit near +-19 in real units.  The only rounding left is that of
    the split partials and of the bf16 output."""
    import dataclasses
    w = workloads.make_batch("flat_big_v", [64, 40], [4096, 1700], 16, 2,
                             seed=seed)
    kv = w.kv.clone()
    kv[..., :D] = 0x30                      # E4M3 0.5 everywhere
    rng = np.random.default_rng(seed + 100)
    mag = np.clip(300.0 + 60.0 * rng.standard_normal(tuple(kv.shape[:-1]) + (D,)),
                  200.0, 440.0)
    sign = np.where(rng.random(D) < 0.5, -1.0, 1.0)
    v = torch.as_tensor((mag * sign).astype(np.float32)).to(torch.float8_e4m3fn)
    kv[..., D:] = v.view(torch.uint8)
    return dataclasses.replace(w, kv=kv, v_scale=1.0 / 16.0)


def _close(a, b, tol):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), "finite pattern differs"
    err = np.abs(np.where(fin, a, 0) - np.where(fin, b, 0)).max(initial=0.0)
    assert err <= tol, "max abs difference %g > %g" % (err, tol)


# ----------------------------------------------------------------------------

def check_e4m3(lib):
    """All 256 codes decode like torch.float8_e4m3fn, and the printed values
    of the format definition (tests/golden/e4m3_ocp.txt) hold."""
    ours = np.array([lib.oracle_e4m3_decode(c) for c in range(256)])
    ref = _dec_torch(np.arange(256))
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])
    assert np.array_equal(np.signbit(ours[m]), np.signbit(ref[m]))
    path = os.path.join(os.path.dirname(__file__), "golden", "e4m3_ocp.txt")
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code, val = line.split()
        got = lib.oracle_e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val) and \
                math.copysign(1, got) == math.copysign(1, float(val)), code


def check_dense_equivalence(lib):
    """With every visible page selected, the oracle equals dense causal
    attention computed by torch SDPA in float64."""
    for w in small_dense_workloads():
        out, lse, _ = orc.attention(w, lib=lib)
        ref = _sdpa_reference(w)
        _close(out, ref, 1e-12)


def check_brute_force(lib):
    """C oracle == numpy brute force on tiny inputs (with invalid entries)."""
    for seed in (3, 4):
        w = tiny_sparse_workload(seed)
        out, lse, _ = orc.attention(w, lib=lib)
        bo, bl = orc.brute_force_attention(w)
        _close(out, bo, 1e-12)
        _close(lse, bl, 1e-12)


def check_block_table_permutation(lib):
    """Permuting the page pool together with block_table leaves the output
    bit-for-bit unchanged."""
    w = workloads.make_batch("perm", [40, 20], [3000, 700], 8, 2, seed=5)
    out, lse, _ = orc.attention(w, lib=lib)
    g = torch.Generator().manual_seed(9)
    perm = torch.randperm(w.num_pages, generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(w.num_pages)
    kv2 = w.kv[perm]                      # new page i = old page perm[i]
    bt2 = torch.where(w.block_table >= 0, inv[w.block_table.long().clamp(min=0)]
                      .to(torch.int32), w.block_table)
    out2, lse2, _ = orc.attention(_replace(w, kv=kv2, block_table=bt2), lib=lib)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def check_padding_and_order(lib):
    """Reordering a token's list, repeating a listed page, or turning a
    repeat into -1 padding leaves the output unchanged."""
    w = workloads.make_batch("pad", [48], [2500], 8, 2, seed=6)
    out, lse, _ = orc.attention(w, lib=lib)
    g = torch.Generator().manual_seed(1)
    tk = w.topk.clone()
    for t in range(tk.shape[0]):
        for h in range(tk.shape[1]):
            tk[t, h] = tk[t, h][torch.randperm(16, generator=g)]
    out2, lse2, _ = orc.attention(_replace(w, topk=tk), lib=lib)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    # a token with fewer than 16 visible pages: replace its -1 entries with
    # repeats of its first entry
    w3 = workloads.make_batch("pad3", [40], [700], 8, 2, seed=7)
    o3, l3, _ = orc.attention(w3, lib=lib)
    tk3 = w3.topk.clone()
    first = tk3[..., :1].expand_as(tk3)
    tk3 = torch.where(tk3 < 0, first, tk3)
    o4, l4, _ = orc.attention(_replace(w3, topk=tk3), lib=lib)
    assert np.array_equal(o3, o4) and np.array_equal(l3, l4)


def check_closed_forms(lib):
    """(1) The first token of a sequence sees only key 0: out = dec(V0)*s_v
    exactly and lse = its score.  (2) Constant V gives out = V.  (3) Zero Q
    gives the plain mean of the attended V rows and lse = ln(#keys).
    (4) #keys = 15*128 + pos%128 + 1 for a token whose 16 valid pages are
    distinct and include its own page; pos + 1 when all its pages are
    selected."""
    w = workloads.make_batch("cf", [300], [300], 8, 2, seed=8)
    out, lse, nk = orc.attention(w, tokens=[0], lib=lib)
    qd = _dec_torch(w.q.numpy()) * w.q_scale
    kvd = _dec_torch(w.kv.numpy())
    phys0 = int(w.block_table[0, 0])
    for hq in range(w.Hq):
        h = hq // w.G
        v0 = kvd[phys0, h, 0, D:] * w.v_scale
        k0 = kvd[phys0, h, 0, :D] * w.k_scale
        assert np.array_equal(out[0, hq], v0)
        s = float(np.dot(qd[0, hq], k0)) * w.softmax_scale
        assert abs(lse[0, hq] - s) <= 1e-12 * max(1.0, abs(s))
    assert (nk[0] == 1).all()

    # constant V
    kv = w.kv.clone()
    kv[..., D:] = 0x3A                            # 1.25
    o2, _, _ = orc.attention(_replace(w, kv=kv), lib=lib)
    assert np.abs(o2 - 1.25 * w.v_scale).max() < 1e-12

    # zero Q: uniform weights over the attended keys
    w5 = workloads.make_batch("zq", [64, 32], [2600, 200], 4, 2, seed=10)
    q0 = torch.zeros_like(w5.q)
    o5, l5, n5 = orc.attention(_replace(w5, q=q0), lib=lib)
    kvd5 = _dec_torch(w5.kv.numpy())
    tk = w5.topk.numpy()
    for t in (0, 17, 63, 64, 95):
        b = 0 if t < 64 else 1
        i = t - int(w5.cu_q[b])
        sl, ql = w5.seq_lens[b], w5.q_lens[b]
        pos = sl - ql + i
        npg = (sl + PAGE - 1) // PAGE
        for h in range(w5.Hkv):
            pages = sorted({int(p) for p in tk[t, h] if 0 <= p < npg})
            keys = [p * PAGE + k for p in pages for k in range(PAGE)
                    if p * PAGE + k <= pos]
            rows = np.array([kvd5[int(w5.block_table[b, k // PAGE]), h,
                                  k % PAGE, D:] for k in keys]) * w5.v_scale
            for g in range(w5.G):
                hq = h * w5.G + g
                assert np.abs(o5[t, hq] - rows.mean(0)).max() < 1e-12
                assert abs(l5[t, hq] - math.log(len(keys))) < 1e-12
            own = pos // PAGE
            if len(pages) == 16 and own in pages:
                assert n5[t, h] == 15 * PAGE + pos % PAGE + 1
            if len(pages) == own + 1:
                assert n5[t, h] == pos + 1


def check_combine_identity(lib):
    """Attending over two disjoint halves of each token's page list and
    merging the halves by log-sum-exp equals attending over the whole list;
    merging a single slot is the identity; two equal slots keep O and add
    ln 2 to lse."""
    w = workloads.make_batch("split", [24, 16], [4000, 2100], 8, 2, seed=11)
    full_o, full_l, _ = orc.attention(w, lib=lib)
    tk = w.topk.clone()
    a = tk.clone()
    a[..., 8:] = -1
    b = tk.clone()
    b[..., :8] = -1
    oa, la, _ = orc.attention(_replace(w, topk=a), lib=lib)
    ob, lb, _ = orc.attention(_replace(w, topk=b), lib=lib)
    po = np.stack([oa, ob], axis=2).reshape(-1, 2, D)
    pl = np.stack([la, lb], axis=2).reshape(-1, 2)
    mo, ml = orc.combine(po, pl, lib=lib)
    _close(mo.reshape(full_o.shape), full_o, 1e-12)
    _close(ml.reshape(full_l.shape), full_l, 1e-12)
    one_o, one_l = orc.combine(po[:, :1], pl[:, :1], lib=lib)
    assert np.array_equal(one_o, po[:, 0]) and np.array_equal(one_l, pl[:, 0])
    two = np.concatenate([po[:, :1], po[:, :1]], 1)
    tl = np.concatenate([pl[:, :1], pl[:, :1]], 1)
    t_o, t_l = orc.combine(two, tl, lib=lib)
    _close(t_o, po[:, 0], 1e-12)
    _close(t_l, pl[:, 0] + math.log(2.0), 1e-12)
    e_o, e_l = orc.combine(np.zeros((2, 3, D)), np.full((2, 3), -np.inf),
                           lib=lib)
    assert (e_o == 0).all() and np.isneginf(e_l).all()


def python_loop_inversion(w, total_rows=None):
    """The CSR as a plain dict of lists: walk tokens in ascending order and
    append each valid, first-seen, not-future page to its row."""
    tk = w.topk.numpy()
    bt = w.block_table.numpy()
    R = w.total_rows if total_rows is None else total_rows
    rows = {}
    mask = np.zeros((w.T, w.Hkv), np.uint16)
    off = 0
    for b in range(w.B):
        ql, sl = w.q_lens[b], w.seq_lens[b]
        npg = (sl + PAGE - 1) // PAGE
        for i in range(ql):
            t = int(w.cu_q[b]) + i
            own = (sl - ql + i) // PAGE
            for h in range(w.Hkv):
                seen = set()
                for j in range(16):
                    p = int(tk[t, h, j])
                    if p in seen:
                        continue
                    seen.add(p)
                    if not (0 <= p < npg) or p > own:
                        continue
                    if not (0 <= bt[b, p] < w.num_pages):
                        continue
                    rows.setdefault(h * R + off + p, []).append((t, j))
                    mask[t, h] |= 1 << j
        off += npg
    return rows, mask


def check_csr(lib):
    """The oracle's CSR equals the dict-of-lists inversion, row by row; rows
    are ascending in token id; counts add up to the kept entries."""
    for w in (tiny_sparse_workload(3), tiny_sparse_workload(4),
              workloads.make_config("ragged_batch_8", seed=0)):
        row_ptr, q_idx, slot, mask = orc.k2q_csr(w, lib=lib)
        rows, mask_ref = python_loop_inversion(w)
        nrows = w.Hkv * w.total_rows
        assert len(row_ptr) == nrows + 1 and row_ptr[0] == 0
        assert (np.diff(row_ptr) >= 0).all()
        assert row_ptr[-1] == sum(len(v) for v in rows.values())
        for r in range(nrows):
            got = list(zip(q_idx[row_ptr[r]:row_ptr[r + 1]].tolist(),
                           slot[row_ptr[r]:row_ptr[r + 1]].tolist()))
            assert got == rows.get(r, []), r
        assert np.array_equal(mask, mask_ref)


def check_e4m3_encode(lib):
    """The E4M3 encoder (nearest, ties to even, saturating at 448) against
    the format's own codes and against torch's float8_e4m3fn cast: every
    finite code encodes back to itself; random values and the exact
    midpoints between neighbouring codes round as torch rounds them; values
    past 448 saturate."""
    dec = [lib.oracle_e4m3_decode(c) for c in range(256)]
    for c, v in enumerate(dec):
        if not math.isnan(v):
            assert lib.oracle_e4m3_encode(v) == c, hex(c)
    pos = sorted({v for v in dec if not math.isnan(v) and v >= 0})
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    rng = np.random.default_rng(21)
    xs = np.concatenate([mids, [-m for m in mids],
                         rng.standard_normal(2000) * 40.0,
                         rng.uniform(-0.02, 0.02, 500)])
    xs = xs[np.abs(xs) < 448.0]
    want = torch.as_tensor(xs.astype(np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()
    got = np.array([lib.oracle_e4m3_encode(float(np.float32(x))) for x in xs])
    assert np.array_equal(got, want)
    for x, c in ((449.0, 0x7E), (1e6, 0x7E), (-500.0, 0xFE)):
        assert lib.oracle_e4m3_encode(x) == c


def check_nvfp4(lib):
    """E2M1 decoding against the format definition
    (tests/golden/e2m1_ocp.txt); the NVFP4 -> E4M3 conversion of a slot with
    random codes and block scales against a restatement here: the nibble of
    element e is byte e // 2 (low nibble first), its scale is scale e // 16
    of its token, and the product is rounded by torch's float8_e4m3fn cast."""
    path = os.path.join(os.path.dirname(__file__), "golden", "e2m1_ocp.txt")
    table = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code, val = line.split()
        got = lib.oracle_e2m1_decode(int(code, 16))
        assert got == float(val) and \
            math.copysign(1, got) == math.copysign(1, float(val)), code
        table[int(code, 16)] = float(val)
    rng = np.random.default_rng(22)
    slot = 128 * 64 + 128 * 8
    kv4 = np.zeros((3, 1, 2, slot), np.uint8)
    kv4[..., :128 * 64] = rng.integers(0, 256, size=(3, 1, 2, 128 * 64))
    # block scales: E4M3 codes of magnitudes up to 74 (code times scale stays
    # within 448), zero included
    kv4[..., 128 * 64:] = rng.integers(0, 0x6A, size=(3, 1, 2, 128 * 8))
    out = np.zeros((3, 1, 128, 256), np.uint8)
    lib.oracle_nvfp4_to_e4m3(kv4.ctypes.data_as(ctypes.c_void_p), 3,
                             out.ctypes.data_as(ctypes.c_void_p))
    codes = kv4[..., :128 * 64].reshape(3, 1, 2, 128, 64)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(3, 1, 2, 128, 128)
    vals = np.vectorize(table.get)(nib).astype(np.float64)
    sc = _dec_torch(kv4[..., 128 * 64:].reshape(3, 1, 2, 128, 8))
    prod = vals * np.repeat(sc, 16, axis=-1)
    want = torch.as_tensor(prod.astype(np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()
    want = np.concatenate([want[:, :, 0], want[:, :, 1]], axis=-1)  # K | V
    assert np.array_equal(out, want)


def check_bf16(lib):
    """All 65536 bfloat16 codes decode like torch's bfloat16 -> float64 cast
    (NaN codes to NaN, signed zeros and infinities included)."""
    codes = np.arange(65536, dtype=np.uint32)
    ours = np.array([lib.oracle_bf16_decode(int(c)) for c in codes])
    ref = torch.from_numpy(codes.astype(np.int32).astype(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])
    assert np.array_equal(np.signbit(ours[m]), np.signbit(ref[m]))


def check_bf16_query(lib):
    """The BF16-query attention ([P2] Details: BF16-Q x FP8-K/V): (1) given
    the E4M3 query widened to bfloat16 (exact: every E4M3 value is a
    bfloat16 value) and the same q_scale, it returns the E4M3-query result
    bit for bit, on a batch with invalid entries; (2) with a BF16 query of
    N(0,1) values (not E4M3 values) and every visible page selected, it
    equals dense causal attention by torch SDPA in float64; (3) it equals
    the numpy brute force on tiny inputs."""
    w = tiny_sparse_workload(3)
    out, lse, nk = orc.attention(w, lib=lib)
    q16 = torch.from_numpy(_dec_torch(w.q.numpy())).to(torch.bfloat16)
    assert np.array_equal(q16.to(torch.float64).numpy(), _dec_torch(w.q.numpy()))
    o2, l2, n2 = orc.attention(_replace(w, q=None, q16=q16), lib=lib)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2) and \
        np.array_equal(nk, n2)
    for wd in small_dense_workloads():
        wb = workloads.with_bf16_query(wd, seed=4)
        ob, _, _ = orc.attention(wb, lib=lib)
        _close(ob, _sdpa_reference(wb), 1e-12)
    for seed in (3, 4):
        wb = workloads.with_bf16_query(tiny_sparse_workload(seed), seed=seed)
        ob, lb, _ = orc.attention(wb, lib=lib)
        bo, bl = orc.brute_force_attention(wb)
        _close(ob, bo, 1e-12)
        _close(lb, bl, 1e-12)


def schedule_cases():
    """(workload, total_rows) pairs for the work-list pins: GQA groups from
    1 to 128 (chunks of 128 down to 1 token), ragged batches with two KV
    heads, spare rows past the requests' pages, invalid entries, and rows
    selected by hundreds of tokens (many chunks per row)."""
    cases = []
    for hq, hkv, seed in ((16, 2, 31), (3, 1, 32), (12, 4, 33), (128, 1, 34),
                          (4, 4, 35)):
        w = workloads.make_batch("sched", [300, 40, 7], [2000, 900, 7], hq,
                                 hkv, seed=seed)
        cases.append((w, w.total_rows))
    w = workloads.make_batch("sched_long", [1500], [1500], 16, 2, seed=36)
    cases.append((w, w.total_rows + 5))
    w = tiny_sparse_workload(3)
    cases.append((w, w.total_rows))
    return cases


def check_schedule(schedule=None):
    """The work list against what its rule fixes, from a CSR built by the
    plain Python inversion (not the oracle's): every item's token count n
    satisfies 1 <= n and n * G <= 128 (one 128-row MMA tile of n tokens x G
    query heads); the items' CSR ranges lie inside their own row
    (h * R + request offset + p) and, taken in order, tile [0, nnz) exactly
    once, so rows come in ascending order; every item of a row but its last
    is full (floor(128 / G) tokens); a row of c entries gives
    ceil(c / floor(128 / G)) items."""
    schedule = schedule or orc.schedule
    for w, R in schedule_cases():
        rows, _ = python_loop_inversion(w, total_rows=R)
        nrows = w.Hkv * R
        cnt = np.zeros(nrows, np.int64)
        for r, v in rows.items():
            cnt[r] = len(v)
        row_ptr = np.zeros(nrows + 1, np.int64)
        row_ptr[1:] = np.cumsum(cnt)
        off = np.zeros(w.B + 1, np.int64)
        off[1:] = np.cumsum(w.pages_per_request)
        full = 128 // w.G
        items = schedule(row_ptr, w, total_rows=R)
        at, last_row = 0, -1
        per_row = {}
        for start, n, b, h, p in items:
            assert 1 <= n and n * w.G <= 128, (n, w.G)
            assert 0 <= b < w.B and 0 <= h < w.Hkv and \
                0 <= p < w.pages_per_request[b]
            r = h * R + int(off[b]) + p
            assert row_ptr[r] <= start and start + n <= row_ptr[r + 1], (r, start)
            assert start == at, "items do not tile the CSR in order"
            assert r >= last_row, "rows out of order"
            at, last_row = start + n, r
            per_row.setdefault(r, []).append(n)
        assert at == row_ptr[-1]
        assert len(items) == sum(-(-int(c) // full) for c in cnt)
        for r, ns in per_row.items():
            assert all(n == full for n in ns[:-1]), r
            assert sum(ns) == cnt[r]


ALL_CHECKS = [check_e4m3, check_dense_equivalence, check_brute_force,
              check_block_table_permutation, check_padding_and_order,
              check_closed_forms, check_combine_identity, check_csr,
              check_e4m3_encode, check_nvfp4, check_bf16, check_bf16_query]
