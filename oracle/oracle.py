"""Python side of the FP64 oracle (TEST INFRASTRUCTURE ONLY).

The heavy loops live in ``msa_oracle.c`` (plain C, FP64, OpenMP over
(token, KV head)); this module loads it with ctypes and adds two pieces that
are small enough to state in Python: the work-list rule and a numpy brute
force used to pin the C code on tiny inputs.

Citations use the pages' addresses:
  [P2] vLLM PR 60684 "MSA prefill takes the E4M3 query natively"
  [P4] vLLM docs, minimax_m3/nvidia/sparse_attention_msa,
       MiniMaxM3SparseMSAImpl.forward
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

D = 128
PAGE = 128
TOPK = 16

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        _lib_setup(lib)
        _lib = lib
    return _lib


def load_library(path: str):
    """Load an oracle library built from another source file (the pin tests
    build planted-mistake copies this way); pass it as ``lib=`` to the
    functions below."""
    lib = ctypes.CDLL(path)
    _lib_setup(lib)
    return lib


def _lib_setup(lib):
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = f64
    lib.oracle_attention.argtypes = [P, P, i64, P, P, i32, P, P, i32, i32,
                                     i32, f64, f64, f64, f64, P, i64, P, P, P,
                                     i32]
    lib.oracle_attention.restype = i32
    lib.oracle_attention_bf16q.argtypes = lib.oracle_attention.argtypes
    lib.oracle_attention_bf16q.restype = i32
    lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_decode.restype = f64
    lib.oracle_k2q_csr.argtypes = [P, P, i32, i64, P, P, i32, i32, i64, P, P,
                                   P, i64, P]
    lib.oracle_k2q_csr.restype = i64
    lib.oracle_combine.argtypes = [P, P, i64, i32, i32, P, P]
    lib.oracle_combine.restype = None
    lib.oracle_max_threads.restype = i32
    lib.oracle_e4m3_encode.argtypes = [f64]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1_decode.restype = f64
    lib.oracle_nvfp4_to_e4m3.argtypes = [P, i64, P]
    lib.oracle_nvfp4_to_e4m3.restype = None


def _np(x, dtype):
    """Contiguous numpy copy of a torch tensor or array with ``dtype``."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=dtype)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """The uint16 codes of a torch bfloat16 tensor (or a uint16 array)."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(np.asarray(x).view(np.uint16))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def e4m3_decode(code: int) -> float:
    """OCP E4M3 (FN) decoding, from the format definition (bias 7)."""
    return float(_load().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def bf16_decode(code: int) -> float:
    """bfloat16 decoding, from the format definition (bias 127)."""
    return float(_load().oracle_bf16_decode(int(code) & 0xFFFF))


def e4m3_encode(x: float) -> int:
    """Nearest E4M3 code (ties to even, saturating at 448), from the format
    definition."""
    return int(_load().oracle_e4m3_encode(float(x)))


def e2m1_decode(code: int) -> float:
    """OCP E2M1 (FP4) decoding, from the format definition (bias 1)."""
    return float(_load().oracle_e2m1_decode(int(code) & 0xF))


def nvfp4_to_e4m3(kv4, lib=None) -> np.ndarray:
    """The E4M3 pool an E4M3-query kernel reads from an NVFP4 pool ([P2]
    vLLM PR 60684, Details: each code times its block scale, dequantised to
    E4M3): uint8 [pages][Hkv][2][slot bytes] -> uint8 [pages][Hkv][128][256]."""
    lib = lib or _load()
    k4 = _np(kv4, np.uint8)
    pages, hkv = int(k4.shape[0]), int(k4.shape[1])
    kv8 = np.zeros((pages, hkv, PAGE, 2 * D), np.uint8)
    lib.oracle_nvfp4_to_e4m3(_ptr(k4), pages * hkv, _ptr(kv8))
    return kv8


def attention(w, tokens=None, nthreads: int = 0, lib=None):
    """Masked softmax attention of ``w`` (a ``workloads.Workload``) in FP64.

    For request b, local query i and global token t: position
    pos = seq_len_b - q_len_b + i ([P2] Performance: chunks sit at the tail);
    key set = every key k of a selected page (logical id in [0, P_b), mapped
    through block_table) with k <= pos and k < seq_len_b ([P4]: causal=True,
    seqused_k); score = (dec(Q) q_scale) . (dec(K) k_scale) * softmax_scale;
    out = softmax-weighted sum of dec(V) v_scale; lse = ln sum exp(score).
    A workload with a BF16 query (``w.q16``, [P2] Details: the BF16-Q x
    FP8-K/V mode) takes bf16(Q) q_scale for dec(Q) q_scale.

    Returns (out [n, Hq, 128], lse [n, Hq], nkeys [n, Hkv]) for the listed
    tokens (all when ``tokens`` is None).
    """
    lib = lib or _load()
    q16 = getattr(w, "q16", None)
    q = _bf16_bits(q16) if q16 is not None else _np(w.q, np.uint8)
    fn = lib.oracle_attention_bf16q if q16 is not None else lib.oracle_attention
    # an NVFP4 workload is attended over the E4M3 pool its kernel reads; its
    # k_scale / v_scale are the global scales
    kv = nvfp4_to_e4m3(w.kv4, lib) if w.kv is None else _np(w.kv, np.uint8)
    topk = _np(w.topk, np.int32)
    bt = _np(w.block_table, np.int32)
    cu_q = _np(w.cu_q, np.int32)
    cu_k = _np(w.cu_k, np.int32)
    T = int(cu_q[-1]) if len(cu_q) else 0
    if tokens is None:
        tok = None
        n = T
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        n = len(tok)
    out = np.zeros((n, w.Hq, D), np.float64)
    lse = np.zeros((n, w.Hq), np.float64)
    nk = np.zeros((n, w.Hkv), np.int32)
    bt_stride = bt.shape[1] if bt.ndim == 2 else 1
    rc = fn(
        _ptr(q), _ptr(kv), int(kv.shape[0]), _ptr(topk), _ptr(bt), bt_stride,
        _ptr(cu_q), _ptr(cu_k), w.B, w.Hq, w.Hkv, float(w.q_scale),
        float(w.k_scale), float(w.v_scale), float(w.softmax_scale),
        _ptr(tok) if tok is not None else None, n, _ptr(out), _ptr(lse),
        _ptr(nk), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attention: a token belongs to no request")
    return out, lse, nk


def k2q_csr(w, total_rows=None, lib=None):
    """Page-to-query CSR by plain loops ([P4] build_k2q_csr).

    Returns (row_ptr [Hkv*R+1], q_idx [nnz], slot [nnz], slot_mask [T, Hkv])
    with R = ``total_rows`` (default: the sum of the requests' page counts).
    """
    lib = lib or _load()
    topk = _np(w.topk, np.int32)
    bt = _np(w.block_table, np.int32)
    cu_q = _np(w.cu_q, np.int32)
    cu_k = _np(w.cu_k, np.int32)
    R = int(w.total_rows if total_rows is None else total_rows)
    rows = w.Hkv * R
    T = int(cu_q[-1]) if len(cu_q) else 0
    cap = max(1, T * w.Hkv * TOPK)
    row_ptr = np.zeros(rows + 1, np.int32)
    q_idx = np.zeros(cap, np.int32)
    slot = np.zeros(cap, np.uint8)
    mask = np.zeros((max(T, 1), w.Hkv), np.uint16)
    bt_stride = bt.shape[1] if bt.ndim == 2 else 1
    nnz = lib.oracle_k2q_csr(_ptr(topk), _ptr(bt), bt_stride,
                             int(w.num_pages), _ptr(cu_q), _ptr(cu_k), w.B,
                             w.Hkv, R, _ptr(row_ptr), _ptr(q_idx), _ptr(slot),
                             cap, _ptr(mask))
    if nnz < 0:
        raise ValueError("oracle_k2q_csr failed (%d)" % nnz)
    return row_ptr, q_idx[:nnz].copy(), slot[:nnz].copy(), mask[:T].copy()


def schedule(row_ptr, w, total_rows=None):
    """The work list, stated directly: rows in ascending order, each row cut
    into chunks of C = 128 // G consecutive CSR entries (C tokens x G query
    heads fill the 128 rows of one tile).  Each item is
    (start, count, b, h, p): CSR offset, tokens, request, KV head, logical
    page.  This rule is this library's own (the pages show a schedule object
    but not its contents)."""
    R = int(w.total_rows if total_rows is None else total_rows)
    C = 128 // w.G
    off = np.zeros(w.B + 1, np.int64)
    off[1:] = np.cumsum(w.pages_per_request)
    items = []
    for h in range(w.Hkv):
        for b in range(w.B):
            for p in range(w.pages_per_request[b]):
                r = h * R + int(off[b]) + p
                a, e = int(row_ptr[r]), int(row_ptr[r + 1])
                for c in range(a, e, C):
                    items.append((c, min(C, e - c), b, h, p))
    return items


def combine(part_o, part_lse, lib=None):
    """Log-sum-exp merge of split partials in FP64.

    part_o [rows, S, D] (each O_j already normalised), part_lse [rows, S]
    with -inf marking an empty slot.  Returns (out [rows, D], lse [rows])."""
    lib = lib or _load()
    po = _np(part_o, np.float64)
    pl = _np(part_lse, np.float64)
    rows, S, Dd = po.shape
    out = np.zeros((rows, Dd), np.float64)
    lse = np.zeros(rows, np.float64)
    lib.oracle_combine(_ptr(po), _ptr(pl), rows, S, Dd, _ptr(out), _ptr(lse))
    return out, lse


def brute_force_attention(w):
    """Numpy triple loop for tiny inputs, written independently of the C code:
    for every (token, query head) it walks *all* keys 0..seq_len-1 of the
    request and keeps a key when its page appears among the token's valid
    top-k entries and the key is not after the query.  E4M3 decoding here is
    torch's float8_e4m3fn cast (a library routine), not the oracle's table;
    a BF16 query (``w.q16``) is widened by torch's bfloat16 cast."""
    import torch

    def dec(x):
        t = torch.as_tensor(np.asarray(x, dtype=np.uint8))
        return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()

    q16 = getattr(w, "q16", None)
    q = (q16.to(torch.float64).numpy() if q16 is not None
         else dec(_np(w.q, np.uint8)))
    kv = dec(_np(w.kv, np.uint8))
    topk = _np(w.topk, np.int32)
    bt = _np(w.block_table, np.int32)
    cu_q = _np(w.cu_q, np.int64)
    cu_k = _np(w.cu_k, np.int64)
    G = w.Hq // w.Hkv
    T = int(cu_q[-1])
    out = np.zeros((T, w.Hq, D))
    lse = np.full((T, w.Hq), -np.inf)
    for b in range(w.B):
        ql = cu_q[b + 1] - cu_q[b]
        sl = cu_k[b + 1] - cu_k[b]
        npg = (sl + PAGE - 1) // PAGE
        for i in range(ql):
            t = cu_q[b] + i
            pos = sl - ql + i
            for hq in range(w.Hq):
                h = hq // G
                chosen = [int(p) for p in topk[t, h]
                          if 0 <= p < npg and 0 <= bt[b, p] < kv.shape[0]]
                scores, vals = [], []
                for k in range(sl):
                    if k // PAGE in chosen and k <= pos:
                        phys = bt[b, k // PAGE]
                        krow = kv[phys, h, k % PAGE, :D] * w.k_scale
                        vrow = kv[phys, h, k % PAGE, D:] * w.v_scale
                        qrow = q[t, hq] * w.q_scale
                        scores.append(float(np.dot(qrow, krow))
                                      * w.softmax_scale)
                        vals.append(vrow)
                if scores:
                    s = np.array(scores)
                    m = s.max()
                    e = np.exp(s - m)
                    out[t, hq] = (e[:, None] * np.array(vals)).sum(0) / e.sum()
                    lse[t, hq] = m + math.log(e.sum())
    return out, lse
