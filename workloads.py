"""Seeded synthetic inputs for MSA block-sparse attention.

This module only draws inputs. It holds no part of the attention arithmetic,
the page-to-query inversion or the split combine, so the CPU oracle (under
``oracle/``) and the CUDA library can both consume what it returns without
sharing any of the method's code.

What it draws follows the per-layer benchmark of vLLM PR 60684 ("MSA prefill
takes the E4M3 query natively", section Performance):

* for every query token and KV head, a uniform random score for each page
  before the token's own page, score 2.0 for the own page, and -1 for pages
  after it; the 16 best-scoring pages are kept, and a kept page whose score is
  negative becomes -1 (padding) -- so a token that sees fewer than 16 pages
  gets all of them plus -1 entries;
* the block table is a random permutation of the physical pages;
* Q, K and V are N(0, 1) in fp32, quantised to OCP E4M3 with one scale per
  tensor, ``amax / 448`` (the values are clamped to +-448 before the cast so
  rounding can never reach the NaN code).

The packed page layout ``[pages, Hkv, 128 tokens, 256 bytes]`` with K in bytes
0..127 and V in bytes 128..255 of each token row is vLLM's packed K|V page, as
the MSA implementation page (vLLM docs, ``MiniMaxM3SparseMSAImpl.forward``)
splits it with ``kv_cache.split(head_size, dim=-1)``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128
PAGE = 128
TOPK = 16
E4M3_MAX = 448.0
E2M1_MAX = 6.0
# NVFP4 page slot (one KV head's K or V of one page): 128 tokens x 64 bytes
# of packed E2M1 codes, then 128 tokens x 8 E4M3 block scales
NVFP4_BLOCK = 16  # elements per E4M3 block scale
NVFP4_SLOT_BYTES = PAGE * (HEAD_DIM // 2) + PAGE * (HEAD_DIM // NVFP4_BLOCK)
SOFTMAX_SCALE = 1.0 / math.sqrt(HEAD_DIM)


@dataclass
class Workload:
    """One batch of prefill (or decode) inputs, all in the library's layouts.

    q           uint8  [T, Hq, 128]            E4M3 codes (None with q16)
    q16         bfloat16 [T, Hq, 128]          a BF16 query, or None
    kv          uint8  [num_pages, Hkv, 128, 256] E4M3 codes, K | V per token
    topk        int32  [T, Hkv, 16]            logical page ids, -1 = padding
    block_table int32  [B, bt_stride]          logical -> physical page, -1 pad
    cu_q, cu_k  int32  [B + 1]                 prefix sums of q_len / seq_len
    """

    name: str
    q_lens: list
    seq_lens: list
    Hq: int
    Hkv: int
    q: torch.Tensor
    kv: torch.Tensor
    topk: torch.Tensor
    block_table: torch.Tensor
    cu_q: torch.Tensor
    cu_k: torch.Tensor
    q_scale: float
    k_scale: float
    v_scale: float
    softmax_scale: float = SOFTMAX_SCALE
    meta: dict = field(default_factory=dict)
    # NVFP4 page pool (uint8 [pages][Hkv][2][NVFP4_SLOT_BYTES]), or None; an
    # NVFP4 workload has no E4M3 pool (kv is None) and its k_scale / v_scale
    # are the global scales
    kv4: torch.Tensor = None
    # BF16 query (torch.bfloat16 [T, Hq, 128]) of the BF16-query mode, or
    # None; such a workload has no E4M3 query (q is None) and q_scale 1
    q16: torch.Tensor = None

    @property
    def B(self) -> int:
        return len(self.q_lens)

    @property
    def T(self) -> int:
        return int(sum(self.q_lens))

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def num_pages(self) -> int:
        return int((self.kv if self.kv is not None else self.kv4).shape[0])

    @property
    def pages_per_request(self) -> list:
        return [(s + PAGE - 1) // PAGE for s in self.seq_lens]

    @property
    def total_rows(self) -> int:
        """Sum over requests of their page counts (vLLM's total_kv_blocks)."""
        return int(sum(self.pages_per_request))

    @property
    def max_seqlen_q(self) -> int:
        return int(max(self.q_lens)) if self.q_lens else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(max(self.seq_lens)) if self.seq_lens else 0

    def to(self, device) -> "Workload":
        """Same workload with every tensor moved to ``device``."""
        mv = {k: (None if getattr(self, k) is None else getattr(self, k).to(device))
              for k in ("q", "kv", "topk", "block_table", "cu_q", "cu_k", "kv4",
                        "q16")}
        return Workload(self.name, list(self.q_lens), list(self.seq_lens),
                        self.Hq, self.Hkv, q_scale=self.q_scale,
                        k_scale=self.k_scale, v_scale=self.v_scale,
                        softmax_scale=self.softmax_scale, meta=dict(self.meta),
                        **mv)


# ----------------------------------------------------------------------------
# random streams
# ----------------------------------------------------------------------------

def _streams(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s))
            for s in np.random.SeedSequence(seed).spawn(n)]


def _quantize(x: torch.Tensor, scale: float) -> torch.Tensor:
    return (x / scale).clamp_(-E4M3_MAX, E4M3_MAX).to(
        torch.float8_e4m3fn).view(torch.uint8)


def _normal_chunks(rng_seed: int, shape, device="cpu"):
    """N(0,1) fp32 of ``shape`` drawn in chunks along axis 0: yields
    (start, stop, chunk).  The same seed gives the same numbers every time."""
    shape = tuple(int(s) for s in shape)
    n0 = shape[0]
    inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    chunk = max(1, (1 << 26) // max(inner, 1))
    if device == "cpu":
        rng = np.random.Generator(np.random.PCG64(rng_seed))
        for a in range(0, n0, chunk):
            b = min(n0, a + chunk)
            yield a, b, torch.from_numpy(
                rng.standard_normal((b - a,) + shape[1:], dtype=np.float32))
    else:
        g = torch.Generator(device=device)
        g.manual_seed(rng_seed)
        for a in range(0, n0, chunk):
            b = min(n0, a + chunk)
            yield a, b, torch.randn((b - a,) + shape[1:], generator=g,
                                    device=device, dtype=torch.float32)


def _normal_e4m3(rng_seed: int, shape, device="cpu", split_last=None):
    """N(0,1) fp32 of ``shape`` quantised to E4M3 with a per-tensor scale.

    With ``split_last=c`` the last axis is cut at ``c`` and the two parts get
    separate scales (K and V of a packed page).  The draw is made in chunks
    along axis 0 twice (once for amax, once to quantise) so that large pools
    never hold their fp32 copy in memory.
    """
    shape = tuple(int(s) for s in shape)
    parts = [slice(None)] if split_last is None else \
        [slice(0, split_last), slice(split_last, None)]
    amax = [0.0 for _ in parts]
    for _, _, x in _normal_chunks(rng_seed, shape, device):
        for i, sl in enumerate(parts):
            amax[i] = max(amax[i], float(x[..., sl].abs().max()))
    scales = [a / E4M3_MAX if a > 0 else 1.0 for a in amax]
    out = torch.empty(shape, dtype=torch.uint8, device=device)
    for a, b, x in _normal_chunks(rng_seed, shape, device):
        for i, sl in enumerate(parts):
            out[a:b][..., sl] = _quantize(x[..., sl], scales[i])
    return out, scales


_E2M1_VALUES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _e2m1_codes(y: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 value, ties to the even magnitude index; 4-bit codes with
    the sign in bit 3 and the magnitude index in bits 0-2 (input
    generation only)."""
    grid = torch.tensor(_E2M1_VALUES, dtype=torch.float32, device=y.device)
    a = y.abs().clamp(max=E2M1_MAX).contiguous()
    hi = torch.searchsorted(grid, a).clamp(max=7)
    lo = (hi - 1).clamp(min=0)
    dlo, dhi = a - grid[lo], grid[hi] - a
    idx = torch.where((dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0)), hi, lo)
    sign = ((y < 0) & (idx > 0)).to(torch.uint8) << 3
    return idx.to(torch.uint8) | sign


def _nvfp4_slots(x: torch.Tensor, g: float) -> torch.Tensor:
    """fp32 [..., 128 tokens, 128] -> uint8 [..., NVFP4_SLOT_BYTES]: per
    16-element block an E4M3 scale amax / (6 g) and E2M1 codes of x / (scale
    g), two codes per byte with the first in the low nibble."""
    xb = x.reshape(*x.shape[:-1], HEAD_DIM // NVFP4_BLOCK, NVFP4_BLOCK)
    sb = (xb.abs().amax(-1) / (E2M1_MAX * g)).clamp(max=E4M3_MAX).to(
        torch.float8_e4m3fn)
    den = (sb.to(torch.float32) * g).unsqueeze(-1)
    y = torch.where(den > 0, xb / den.clamp(min=1e-30), torch.zeros_like(xb))
    codes = _e2m1_codes(y).reshape(x.shape)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    lead = x.shape[:-2]
    return torch.cat([packed.reshape(*lead, -1),
                      sb.view(torch.uint8).reshape(*lead, -1)], dim=-1)


def _normal_nvfp4(rng_seed: int, num_pages: int, Hkv: int, device="cpu"):
    """The N(0,1) K|V pool of _normal_e4m3 (same draws), quantised to NVFP4
    instead: uint8 [pages][Hkv][2 slots: K, V][NVFP4_SLOT_BYTES] and the
    global scales (K, V) = amax / 448, so that every code times its block
    scale stays within E4M3's range."""
    shape = (num_pages, Hkv, PAGE, 2 * HEAD_DIM)
    amax = [0.0, 0.0]
    for _, _, x in _normal_chunks(rng_seed, shape, device):
        amax[0] = max(amax[0], float(x[..., :HEAD_DIM].abs().max()))
        amax[1] = max(amax[1], float(x[..., HEAD_DIM:].abs().max()))
    gs = [a / E4M3_MAX if a > 0 else 1.0 for a in amax]
    out = torch.empty((num_pages, Hkv, 2, NVFP4_SLOT_BYTES), dtype=torch.uint8,
                      device=device)
    for a, b, x in _normal_chunks(rng_seed, shape, device):
        out[a:b, :, 0] = _nvfp4_slots(x[..., :HEAD_DIM], gs[0])
        out[a:b, :, 1] = _nvfp4_slots(x[..., HEAD_DIM:], gs[1])
    return out, gs


def select_pages(rng, q_len: int, seq_len: int, hkv: int) -> np.ndarray:
    """Top-16 logical page ids per (query token, KV head), -1 padded.

    Query token i of a chunk of ``q_len`` tokens at the tail of ``seq_len``
    sits at position ``seq_len - q_len + i``; its own page is position // 128.
    Scores: U(0,1) for earlier pages, 2.0 for the own page, -1 for later pages.
    """
    out = np.full((q_len, hkv, TOPK), -1, dtype=np.int32)
    if q_len == 0:
        return out
    pos = np.arange(seq_len - q_len, seq_len, dtype=np.int64)
    own = pos // PAGE
    step = max(1, (1 << 24) // max(1, hkv * int(own[-1] + 1)))
    for a in range(0, q_len, step):
        b = min(q_len, a + step)
        o = own[a:b]
        vmax = int(o.max()) + 1
        scores = rng.random((b - a, hkv, vmax), dtype=np.float32)
        ar = np.arange(vmax)[None, None, :]
        oo = o[:, None, None]
        scores = np.where(ar < oo, scores, np.float32(-1.0))
        scores = np.where(ar == oo, np.float32(2.0), scores)
        k = min(TOPK, vmax)
        idx = np.argpartition(-scores, k - 1, axis=-1)[..., :k]
        val = np.take_along_axis(scores, idx, -1)
        order = np.argsort(-val, axis=-1, kind="stable")
        idx = np.take_along_axis(idx, order, -1)
        val = np.take_along_axis(val, order, -1)
        out[a:b, :, :k] = np.where(val >= 0, idx, -1).astype(np.int32)
    return out


def make_batch(name: str, q_lens, seq_lens, Hq: int, Hkv: int, seed: int,
               device="cpu", kv_device=None, extra_pages: int = 0,
               kv_format: str = "e4m3") -> Workload:
    """General prefill batch: request b has ``q_lens[b]`` query tokens at the
    tail of ``seq_lens[b]`` tokens; all requests share one page pool whose
    pages are handed out by a random permutation."""
    q_lens = [int(x) for x in q_lens]
    seq_lens = [int(x) for x in seq_lens]
    assert len(q_lens) == len(seq_lens)
    for ql, sl in zip(q_lens, seq_lens):
        assert 0 <= ql <= sl
    assert Hq % Hkv == 0
    r_top, r_bt, r_q, r_kv = _streams(seed, 4)
    B = len(q_lens)
    pages = [(s + PAGE - 1) // PAGE for s in seq_lens]
    num_pages = int(sum(pages)) + int(extra_pages)
    perm = r_bt.permutation(num_pages).astype(np.int32)
    bt_stride = max(1, max(pages) if pages else 1)
    bt = np.full((max(B, 1), bt_stride), -1, dtype=np.int32)[:B]
    o = 0
    for b in range(B):
        bt[b, :pages[b]] = perm[o:o + pages[b]]
        o += pages[b]
    topk = np.concatenate(
        [select_pages(r_top, ql, sl, Hkv) for ql, sl in zip(q_lens, seq_lens)]
        or [np.zeros((0, Hkv, TOPK), np.int32)], axis=0)
    cu_q = np.zeros(B + 1, np.int32)
    cu_k = np.zeros(B + 1, np.int32)
    cu_q[1:] = np.cumsum(q_lens)
    cu_k[1:] = np.cumsum(seq_lens)
    T = int(cu_q[-1])
    qseed = int(r_q.integers(0, 2**62))
    kvseed = int(r_kv.integers(0, 2**62))
    kvdev = kv_device or device
    q, (qs,) = _normal_e4m3(qseed, (T, Hq, HEAD_DIM), device=device)
    kv4 = None
    if kv_format == "nvfp4":
        kv = None
        kv4, (ks, vs) = _normal_nvfp4(kvseed, num_pages, Hkv, device=kvdev)
    else:
        kv, (ks, vs) = _normal_e4m3(kvseed, (num_pages, Hkv, PAGE, 2 * HEAD_DIM),
                                    device=kvdev, split_last=HEAD_DIM)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return Workload(name, q_lens, seq_lens, Hq, Hkv, q=q, kv=kv,
                    topk=t(topk), block_table=t(bt), cu_q=t(cu_q),
                    cu_k=t(cu_k), q_scale=qs, k_scale=ks, v_scale=vs,
                    meta={"seed": seed, "kv_format": kv_format}, kv4=kv4)


# ----------------------------------------------------------------------------
# the five workloads (the pages' shapes) and their variants
# ----------------------------------------------------------------------------

def ragged_lengths(seed: int, n: int = 8, lo: int = 512, hi: int = 32768,
                   qmin: int = 128, qmax: int = 4096):
    """seq_len log-uniform in [lo, hi]; q_len uniform in
    [qmin, min(seq_len, qmax)] at the tail of the sequence."""
    rng = np.random.Generator(np.random.PCG64(
        np.random.SeedSequence([seed, 7]).generate_state(1)[0]))
    seq = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
    seq = np.clip(np.round(seq).astype(np.int64), lo, hi)
    ql = [int(rng.integers(min(qmin, s), min(s, qmax) + 1)) for s in seq]
    return ql, [int(s) for s in seq]


def decode_lengths(seed: int, n: int, lo: int = 32768, hi: int = 131072):
    rng = np.random.Generator(np.random.PCG64(
        np.random.SeedSequence([seed, 11]).generate_state(1)[0]))
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


CONFIGS = {
    # name: (description, builder(seed, device, kv_device))
    "tiny_full_prefill": "1 request, seq_len = q_len = 1024 (8 pages), "
                         "Hkv=1, Hq=4: every visible page is selected",
    "chunked_prefill_32k": "1 request, q_len 2048 at the tail of 32768 "
                           "tokens (256 pages), Hkv=2, Hq=16",
    "ragged_batch_8": "8 requests, seq_len log-uniform [512, 32768], q_len "
                      "uniform [128, min(seq_len, 4096)], Hkv=2, Hq=16",
    "long_prefill_1m": "1 request, q_len 2048 at the tail of 1,048,576 "
                       "tokens (8192 pages), Hkv=2, Hq=16",
    "long_prefill_150k": "1 request, q_len 8192 at the tail of 153,600 "
                         "tokens (1200 pages), Hkv=2, Hq=16",
    "decode_64x8": "64 requests x 8 query tokens (draft k=7 plus 1), "
                   "seq_len uniform [32768, 131072], Hkv=2, Hq=16",
    "decode_16x8": "16 requests x 8 query tokens, seq_len uniform "
                   "[32768, 131072], Hkv=2, Hq=16",
}


def with_bf16_query(w: Workload, seed: int = 0) -> Workload:
    """The same batch with a BF16 query in place of the E4M3 one: N(0,1)
    values rounded to bfloat16 (nearest even), drawn from a stream of their
    own, so the real query has the scale of the E4M3 workload's
    dec(q) * q_scale; q_scale becomes 1 and q is dropped."""
    import dataclasses
    qseed = int(np.random.SeedSequence([seed, 13]).generate_state(1)[0])
    dev = w.cu_q.device
    q16 = torch.empty((w.T, w.Hq, HEAD_DIM), dtype=torch.bfloat16, device=dev)
    for a, b, x in _normal_chunks(qseed, (w.T, w.Hq, HEAD_DIM), str(dev)):
        q16[a:b] = x.to(torch.bfloat16)
    meta = dict(w.meta)
    meta["query"] = "bf16"
    return dataclasses.replace(w, q=None, q16=q16, q_scale=1.0, meta=meta)


def make_config(name: str, seed: int = 0, device="cpu", kv_device=None):
    """A named workload; a name ending in "_nvfp4" is the same workload with
    an NVFP4 page pool (the same normal draws) instead of the E4M3 one, and
    one ending in "_bf16q" the same workload with a BF16 query."""
    if name.endswith("_bf16q"):
        w = with_bf16_query(make_config(name[:-len("_bf16q")], seed, device,
                                        kv_device), seed)
        w.name = name
        w.meta["description"] += "; BF16 query"
        return w
    if name.endswith("_nvfp4"):
        w = _make_config(name[:-len("_nvfp4")], seed, device, kv_device, "nvfp4")
        w.name = name
        w.meta["description"] += "; NVFP4 K/V pages"
        return w
    return _make_config(name, seed, device, kv_device, "e4m3")


def _make_config(name, seed, device, kv_device, kv_format):
    mb = lambda *a: make_batch(*a, kv_format=kv_format)  # noqa: E731
    if name == "tiny_full_prefill":
        w = mb(name, [1024], [1024], 4, 1, seed, device, kv_device)
    elif name == "chunked_prefill_32k":
        w = mb(name, [2048], [32768], 16, 2, seed, device, kv_device)
    elif name == "ragged_batch_8":
        ql, sl = ragged_lengths(seed)
        w = mb(name, ql, sl, 16, 2, seed, device, kv_device)
    elif name == "long_prefill_1m":
        w = mb(name, [2048], [1048576], 16, 2, seed, device, kv_device)
    elif name == "long_prefill_150k":
        w = mb(name, [8192], [153600], 16, 2, seed, device, kv_device)
    elif name in ("decode_64x8", "decode_16x8"):
        n = 64 if name == "decode_64x8" else 16
        sl = decode_lengths(seed, n)
        w = mb(name, [8] * n, sl, 16, 2, seed, device, kv_device)
    else:
        raise KeyError(name)
    w.meta["description"] = CONFIGS[name]
    return w
