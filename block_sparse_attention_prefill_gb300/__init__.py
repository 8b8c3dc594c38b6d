"""MSA block-sparse attention for GB300: Python binding of libmsa.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of ``libmsa.so`` (see ``include/msa.h`` for the C ABI); PyTorch is
used here for device memory (tensors, workspaces) and the current stream.
There is no fallback: if the library cannot be built or loaded, every call
raises.

Calls (same names as the C ABI, without the ``msa_`` prefix where noted):
  msa_plan      build_k2q_csr + work list on the device
  msa_prefill   sparse attention + log-sum-exp combine -> bf16 out, fp32 lse
  msa_decode    1..8 query tokens per request (decode / speculative verify)
  msa_combine   merge split partials by log-sum-exp
  msa_prefill_nvfp4, msa_decode_nvfp4   the same over NVFP4 K/V pages
  msa_nvfp4_to_e4m3   NVFP4 pages -> the E4M3 pages those calls read
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

HEAD_DIM = 128
PAGE_SIZE = 128
NVFP4_SLOT_BYTES = 9216      # 128 x 64 code bytes + 128 x 8 block scales
TOPK = 16

DTYPE_F32 = 0
DTYPE_BF16 = 1

STATUS_BAD_PAGE_ID = 1 << 0
STATUS_BAD_BLOCK = 1 << 1
STATUS_BAD_SEQLENS = 1 << 2
STATUS_ROWS_OVERFLOW = 1 << 3
STATUS_TIMEOUT = 1 << 4
STATUS_BAD_WORK = 1 << 5

_I64 = ("B", "T", "Hq", "Hkv", "total_rows", "max_seqlen_q", "max_seqlen_k",
        "num_pages", "bt_stride", "bitmap_words", "chunk_tokens", "max_nnz",
        "max_work", "rows", "record_bytes")
_PTR = ("cu_seqlens_q", "cu_seqlens_k", "req_off", "bitmap", "word_pre",
        "row_cnt", "row_loc", "tile_state", "row_ptr", "q_idx", "slot", "work",
        "records", "counters", "slot_mask", "status")


class MsaPlanStruct(ctypes.Structure):
    """Mirror of ``msa_plan_t`` (all fields 64-bit)."""
    _fields_ = [(n, ctypes.c_int64) for n in _I64] + \
               [(n, ctypes.c_void_p) for n in _PTR]


class MsaError(RuntimeError):
    pass


_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load libmsa.so (building it with nvcc first if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build()
    lib = ctypes.CDLL(path)
    P, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    SZ = ctypes.POINTER(ctypes.c_size_t)
    PL = ctypes.POINTER(MsaPlanStruct)
    sigs = {
        "msa_version": ([], i32),
        "msa_status_string": ([i32], ctypes.c_char_p),
        "msa_plan_workspace_bytes": ([i64, i64, i64, i64, i64, i64, SZ], i32),
        "msa_plan": ([P, P, P, P, i64, i64, i64, i64, i64, i64, i64, i64, i64,
                      P, ctypes.c_size_t, PL, P], i32),
        "msa_plan_heads": ([P, i64, i64, P, P, P, i64, i64, i64, i64, i64, i64,
                            i64, i64, i64, P, ctypes.c_size_t, PL, P], i32),
        "msa_prefill_workspace_bytes": ([i64, i64, SZ], i32),
        "msa_prefill": ([P, P, i64, f32, f32, f32, f32, P, i64, PL, P,
                         ctypes.c_size_t, P, P, P], i32),
        "msa_prefill_attention": ([P, P, i64, f32, f32, f32, f32, P, i64, PL,
                                   P, ctypes.c_size_t, P], i32),
        "msa_prefill_combine": ([PL, P, ctypes.c_size_t, P, P, P], i32),
        "msa_combine": ([P, i32, P, i64, i64, P, P, P], i32),
        "msa_decode_workspace_bytes": ([i64, i64, i64, i64, i64, SZ], i32),
        "msa_decode": ([P, P, i64, f32, f32, f32, f32, P, P, i64, P, i64, i64,
                        i64, i64, i64, P, ctypes.c_size_t, P, P, PL, P], i32),
        "msa_decode_noalloc": ([P, P, i64, f32, f32, f32, f32, P, P, i64, P,
                                i64, i64, i64, i64, i64, P, P, P], i32),
        "msa_prefill_nvfp4": ([P, P, i64, f32, f32, f32, f32, P, i64, PL, P,
                               ctypes.c_size_t, P, P, P], i32),
        "msa_decode_nvfp4": ([P, P, i64, f32, f32, f32, f32, P, P, i64, P, i64,
                              i64, i64, i64, i64, P, ctypes.c_size_t, P, P, PL,
                              P], i32),
        "msa_nvfp4_to_e4m3": ([P, i64, P, P], i32),
        "msa_prefill_attention_nvfp4": ([P, P, i64, f32, f32, f32, f32, P, i64,
                                         PL, P, ctypes.c_size_t, P], i32),
        "msa_prefill_bf16q": ([P, P, i64, f32, f32, f32, f32, P, i64, PL, P,
                               ctypes.c_size_t, P, P, P], i32),
        "msa_prefill_attention_bf16q": ([P, P, i64, f32, f32, f32, f32, P, i64,
                                         PL, P, ctypes.c_size_t, P], i32),
        "msa_test_set_wait_limit_ns": ([ctypes.c_uint64], i32),
        "msa_read_status": ([PL, ctypes.POINTER(ctypes.c_uint32)], i32),
        "msa_read_counters": ([PL, ctypes.POINTER(ctypes.c_int64),
                               ctypes.POINTER(ctypes.c_int64)], i32),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().msa_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise MsaError("%s: %s (code %d)" % (what, status_string(rc), rc))


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, name, dtypes, device=True):
    if t is None:
        raise MsaError("%s is required" % name)
    if device and not t.is_cuda:
        raise MsaError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise MsaError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if not t.is_contiguous():
        raise MsaError("%s must be contiguous" % name)


_E4M3 = (torch.uint8, torch.float8_e4m3fn)


def _bytes(t):
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


def _workspace(nbytes, device, given):
    if given is not None:
        if given.numel() * given.element_size() < nbytes:
            raise MsaError("workspace too small: %d < %d bytes"
                           % (given.numel() * given.element_size(), nbytes))
        return given
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def plan_workspace_bytes(B, T, Hq, Hkv, total_rows, max_seqlen_q) -> int:
    n = ctypes.c_size_t()
    _check(load().msa_plan_workspace_bytes(B, T, Hq, Hkv, total_rows,
                                           max_seqlen_q, ctypes.byref(n)),
           "msa_plan_workspace_bytes")
    return n.value


def prefill_workspace_bytes(T, Hq) -> int:
    n = ctypes.c_size_t()
    _check(load().msa_prefill_workspace_bytes(T, Hq, ctypes.byref(n)),
           "msa_prefill_workspace_bytes")
    return n.value


def decode_workspace_bytes(B, n, Hq, Hkv, max_seqlen_k) -> int:
    m = ctypes.c_size_t()
    _check(load().msa_decode_workspace_bytes(B, n, Hq, Hkv, max_seqlen_k,
                                             ctypes.byref(m)),
           "msa_decode_workspace_bytes")
    return m.value


class Plan:
    """A plan built by :func:`msa_plan`.  Holds the C struct and keeps the
    tensors it points into alive."""

    def __init__(self, struct, workspace, keep):
        self.struct = struct
        self.workspace = workspace
        self._keep = keep

    def _view(self, name, count, dtype):
        base = self.workspace.data_ptr()
        off = getattr(self.struct, name) - base
        esz = torch.empty(0, dtype=dtype).element_size()
        return self.workspace[off:off + count * esz].view(dtype)

    # device views of the plan (for tests and inspection)
    def row_ptr(self):
        return self._view("row_ptr", self.struct.rows + 1, torch.int32)

    def q_idx(self):
        return self._view("q_idx", self.struct.max_nnz, torch.int32)

    def slot(self):
        return self._view("slot", self.struct.max_nnz, torch.uint8)

    def work(self):
        return self._view("work", 4 * self.struct.max_work,
                          torch.int32).view(-1, 4)

    def records(self):
        n = self.struct.record_bytes // 16
        return self._view("records", self.struct.max_work * n * 4,
                          torch.int32).view(-1, n, 4)

    def slot_mask(self):
        return self._view("slot_mask", self.struct.T * self.struct.Hkv,
                          torch.int16)

    def status(self) -> int:
        """Device status bits (synchronises)."""
        s = ctypes.c_uint32()
        _check(load().msa_read_status(ctypes.byref(self.struct),
                                      ctypes.byref(s)), "msa_read_status")
        return int(s.value)

    def counters(self):
        """(nnz, num_work) (synchronises)."""
        a, b = ctypes.c_int64(), ctypes.c_int64()
        _check(load().msa_read_counters(ctypes.byref(self.struct),
                                        ctypes.byref(a), ctypes.byref(b)),
               "msa_read_counters")
        return int(a.value), int(b.value)


def msa_plan(topk, cu_seqlens_q, cu_seqlens_k, block_table, num_pages, Hq,
             total_rows, max_seqlen_q, max_seqlen_k, workspace=None,
             stream=None, h_begin=None, h_count=None) -> Plan:
    """build_k2q_csr on the device.  topk int32 [T, Hkv, 16]; cu_seqlens_q/k
    int32 [B+1]; block_table int32 [B, bt_stride].  With h_begin / h_count
    (msa_plan_heads) the plan covers KV heads [h_begin, h_begin + h_count) of
    topk, and Hq is the shard's query heads."""
    _need(topk, "topk", (torch.int32,))
    _need(cu_seqlens_q, "cu_seqlens_q", (torch.int32,))
    _need(cu_seqlens_k, "cu_seqlens_k", (torch.int32,))
    _need(block_table, "block_table", (torch.int32,))
    if topk.dim() != 3 or topk.shape[2] != TOPK:
        raise MsaError("topk must be [T, Hkv, 16]")
    T, topk_hkv = int(topk.shape[0]), int(topk.shape[1])
    sharded = h_begin is not None or h_count is not None
    h0 = int(h_begin or 0)
    Hkv = int(h_count) if h_count is not None else topk_hkv - h0
    B = int(cu_seqlens_q.numel()) - 1
    bt_stride = int(block_table.shape[1]) if block_table.dim() == 2 else 1
    need = plan_workspace_bytes(B, T, Hq, Hkv, total_rows, max_seqlen_q)
    ws = _workspace(need, topk.device, workspace)
    st = MsaPlanStruct()
    args = (_ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(block_table), bt_stride,
            int(num_pages), B, T, int(Hq), Hkv, int(total_rows),
            int(max_seqlen_q), int(max_seqlen_k), _ptr(ws), need,
            ctypes.byref(st), _stream(stream))
    if sharded:
        _check(load().msa_plan_heads(_ptr(topk), topk_hkv, h0, *args), "msa_plan_heads")
    else:
        _check(load().msa_plan(_ptr(topk), *args), "msa_plan")
    return Plan(st, ws, (topk, cu_seqlens_q, cu_seqlens_k, block_table))


def head_shard(Hkv, world, rank):
    """(h_begin, h_count): rank's contiguous share of Hkv KV heads when
    `world` ranks split them evenly (tensor parallelism: each rank owns
    Hkv / world KV heads and their query heads; msa_plan(h_begin=,
    h_count=) then plans that shard)."""
    if world < 1 or not 0 <= rank < world or Hkv % world:
        raise MsaError("%d KV heads do not split evenly over %d ranks" % (Hkv, world))
    n = Hkv // world
    return rank * n, n


def _kv_shape(kv, Hkv, fp4):
    if kv is None:
        raise MsaError("%s is required" % ("kv4" if fp4 else "kv"))
    if fp4:
        if kv.dim() != 4 or tuple(kv.shape[1:]) != (Hkv, 2, NVFP4_SLOT_BYTES):
            raise MsaError("kv4 must be uint8 [num_pages, Hkv, 2, %d]"
                           % NVFP4_SLOT_BYTES)
    elif kv.dim() != 4 or tuple(kv.shape[1:]) != (Hkv, PAGE_SIZE, 2 * HEAD_DIM):
        raise MsaError("kv must be [num_pages, Hkv, 128, 256]")


def _need_kv(kv, Hkv, fp4):
    _kv_shape(kv, Hkv, fp4)
    _need(kv, "kv4" if fp4 else "kv", (torch.uint8,) if fp4 else _E4M3)


def _decode_shapes(q, kv, topk, seq_lens, n, fp4, out=None, lse=None):
    """Shape checks of the decode calls, made before any tensor reaches the
    library (which sees only pointers): q [B*n, Hq, 128], topk
    [B*n, Hkv, 16], the pool for Hkv KV heads, and, when given, out
    [B*n, Hq, 128] and lse [B*n, Hq].  Returns (B, Hq, Hkv)."""
    for t, name in ((q, "q"), (topk, "topk"), (seq_lens, "seq_lens")):
        if t is None:
            raise MsaError("%s is required" % name)
    if q.dim() != 3 or q.shape[2] != HEAD_DIM:
        raise MsaError("q must be [B*n, Hq, 128]")
    if topk.dim() != 3 or topk.shape[2] != TOPK:
        raise MsaError("topk must be [B*n, Hkv, 16]")
    B = int(seq_lens.numel())
    Hq, Hkv = int(q.shape[1]), int(topk.shape[1])
    if q.shape[0] != B * n or topk.shape[0] != B * n:
        raise MsaError("q and topk need B*n rows")
    _kv_shape(kv, Hkv, fp4)
    if out is not None and tuple(out.shape) != (B * n, Hq, HEAD_DIM):
        raise MsaError("out must be [B*n, Hq, 128] = %s" % ((B * n, Hq, HEAD_DIM),))
    if lse is not None and tuple(lse.shape) != (B * n, Hq):
        raise MsaError("lse must be [B*n, Hq] = %s" % ((B * n, Hq),))
    return B, Hq, Hkv


def msa_prefill(q, kv, q_scale, k_scale, v_scale, softmax_scale, block_table,
                plan: Plan, workspace=None, out=None, lse=None,
                want_lse=True, stream=None):
    """Sparse attention + combine.  q E4M3 [T, Hq, 128]; kv E4M3
    [num_pages, Hkv, 128, 256].  Returns (out bf16 [T, Hq, 128],
    lse fp32 [T, Hq] or None)."""
    return _prefill("msa_prefill", q, kv, q_scale, k_scale, v_scale,
                    softmax_scale, block_table, plan, workspace, out, lse,
                    want_lse, stream)


def msa_prefill_nvfp4(q, kv4, q_scale, k_scale, v_scale, softmax_scale,
                      block_table, plan: Plan, workspace=None, out=None,
                      lse=None, want_lse=True, stream=None):
    """msa_prefill over an NVFP4 pool: kv4 uint8 [num_pages, Hkv, 2, 9216]
    (per KV head a K slot then a V slot: 128 x 64 code bytes, then 128 x 8
    E4M3 block scales); k_scale / v_scale are the global scales."""
    return _prefill("msa_prefill_nvfp4", q, kv4, q_scale, k_scale, v_scale,
                    softmax_scale, block_table, plan, workspace, out, lse,
                    want_lse, stream)


def msa_prefill_bf16q(q16, kv, q_scale, k_scale, v_scale, softmax_scale,
                      block_table, plan: Plan, workspace=None, out=None,
                      lse=None, want_lse=True, stream=None):
    """msa_prefill with a BF16 query: q16 bf16 [T, Hq, 128] over the E4M3
    pool (K/V widened to bf16, bf16 MMAs); q_scale multiplies the scores
    (1.0 for a query that already carries its scale)."""
    return _prefill("msa_prefill_bf16q", q16, kv, q_scale, k_scale, v_scale,
                    softmax_scale, block_table, plan, workspace, out, lse,
                    want_lse, stream)


def msa_nvfp4_to_e4m3(kv4, out=None, stream=None):
    """NVFP4 pool -> the E4M3 pool [num_pages, Hkv, 128, 256] that the
    NVFP4 attention reads (each code times its block scale, rounded to
    E4M3)."""
    _need(kv4, "kv4", (torch.uint8,))
    if kv4.dim() != 4 or tuple(kv4.shape[2:]) != (2, NVFP4_SLOT_BYTES):
        raise MsaError("kv4 must be uint8 [num_pages, Hkv, 2, %d]"
                       % NVFP4_SLOT_BYTES)
    P, Hkv = int(kv4.shape[0]), int(kv4.shape[1])
    if out is None:
        out = torch.empty((P, Hkv, PAGE_SIZE, 2 * HEAD_DIM),
                          dtype=torch.float8_e4m3fn, device=kv4.device)
    _need(out, "out", _E4M3)
    _check(load().msa_nvfp4_to_e4m3(_ptr(kv4), P * Hkv, _ptr(_bytes(out)),
                                    _stream(stream)), "msa_nvfp4_to_e4m3")
    return out


def _prefill(name, q, kv, q_scale, k_scale, v_scale, softmax_scale,
             block_table, plan, workspace, out, lse, want_lse, stream):
    _need(q, "q", (torch.bfloat16,) if name.endswith("bf16q") else _E4M3)
    _need(block_table, "block_table", (torch.int32,))
    s = plan.struct
    T, Hq = int(s.T), int(s.Hq)
    if tuple(q.shape) != (T, Hq, HEAD_DIM):
        raise MsaError("q must be [T, Hq, 128] = %s" % ((T, Hq, HEAD_DIM),))
    _need_kv(kv, int(s.Hkv), name.endswith("nvfp4"))
    need = prefill_workspace_bytes(T, Hq)
    ws = _workspace(need, q.device, workspace)
    if out is None:
        out = torch.empty((T, Hq, HEAD_DIM), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", (torch.bfloat16,))
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", (torch.float32,))
    bt_stride = int(block_table.shape[1]) if block_table.dim() == 2 else 1
    _check(getattr(load(), name)(_ptr(_bytes(q)), _ptr(_bytes(kv)),
                                 int(kv.shape[0]), float(q_scale),
                                 float(k_scale), float(v_scale),
                                 float(softmax_scale), _ptr(block_table),
                                 bt_stride, ctypes.byref(s), _ptr(ws), need,
                                 _ptr(out), _ptr(lse), _stream(stream)), name)
    return out, lse


def msa_prefill_attention(q, kv, q_scale, k_scale, v_scale, softmax_scale,
                          block_table, plan: Plan, workspace, stream=None):
    """First half of msa_prefill: the attention kernel, partials into
    ``workspace`` (a uint8 CUDA tensor of prefill_workspace_bytes())."""
    return _attention("msa_prefill_attention", q, kv, q_scale, k_scale,
                      v_scale, softmax_scale, block_table, plan, workspace,
                      stream)


def msa_prefill_attention_nvfp4(q, kv4, q_scale, k_scale, v_scale,
                                softmax_scale, block_table, plan: Plan,
                                workspace, stream=None):
    """The attention half of msa_prefill_nvfp4."""
    return _attention("msa_prefill_attention_nvfp4", q, kv4, q_scale, k_scale,
                      v_scale, softmax_scale, block_table, plan, workspace,
                      stream)


def msa_prefill_attention_bf16q(q16, kv, q_scale, k_scale, v_scale,
                                softmax_scale, block_table, plan: Plan,
                                workspace, stream=None):
    """The attention half of msa_prefill_bf16q."""
    return _attention("msa_prefill_attention_bf16q", q16, kv, q_scale, k_scale,
                      v_scale, softmax_scale, block_table, plan, workspace,
                      stream)


def _attention(name, q, kv, q_scale, k_scale, v_scale, softmax_scale,
               block_table, plan, workspace, stream):
    s = plan.struct
    _need(q, "q", (torch.bfloat16,) if name.endswith("bf16q") else _E4M3)
    _need_kv(kv, int(s.Hkv), name.endswith("nvfp4"))
    need = prefill_workspace_bytes(int(s.T), int(s.Hq))
    ws = _workspace(need, q.device, workspace)
    bt_stride = int(block_table.shape[1]) if block_table.dim() == 2 else 1
    _check(getattr(load(), name)(
        _ptr(_bytes(q)), _ptr(_bytes(kv)), int(kv.shape[0]), float(q_scale),
        float(k_scale), float(v_scale), float(softmax_scale),
        _ptr(block_table), bt_stride, ctypes.byref(s), _ptr(ws), need,
        _stream(stream)), name)
    return ws


def msa_prefill_combine(plan: Plan, workspace, out, lse=None, stream=None):
    """Second half of msa_prefill: merge the partials in ``workspace``."""
    s = plan.struct
    need = prefill_workspace_bytes(int(s.T), int(s.Hq))
    _check(load().msa_prefill_combine(ctypes.byref(s), _ptr(workspace), need,
                                      _ptr(out), _ptr(lse), _stream(stream)),
           "msa_prefill_combine")
    return out, lse


def msa_combine(part_o, part_lse, out=None, lse=None, stream=None):
    """part_o [rows, S, 128] fp32 or bf16 (each normalised), part_lse fp32
    [rows, S] with -inf for an empty split.  Returns (out bf16 [rows, 128],
    lse fp32 [rows])."""
    _need(part_o, "part_o", (torch.float32, torch.bfloat16))
    _need(part_lse, "part_lse", (torch.float32,))
    rows, S = int(part_o.shape[0]), int(part_o.shape[1])
    if part_o.dim() != 3 or part_o.shape[2] != HEAD_DIM or \
            tuple(part_lse.shape) != (rows, S):
        raise MsaError("part_o must be [rows, S, 128], part_lse [rows, S]")
    if out is None:
        out = torch.empty((rows, HEAD_DIM), dtype=torch.bfloat16,
                          device=part_o.device)
    if lse is None:
        lse = torch.empty((rows,), dtype=torch.float32, device=part_o.device)
    dt = DTYPE_F32 if part_o.dtype == torch.float32 else DTYPE_BF16
    _check(load().msa_combine(_ptr(part_o), dt, _ptr(part_lse), rows, S,
                              _ptr(out), _ptr(lse), _stream(stream)),
           "msa_combine")
    return out, lse


def msa_decode(q, kv, q_scale, k_scale, v_scale, softmax_scale, topk,
               block_table, seq_lens, n, max_seqlen_k, workspace=None,
               out=None, lse=None, want_lse=True, stream=None):
    """Decode / speculative verify: n query tokens per request at the tail.
    q E4M3 [B*n, Hq, 128]; topk int32 [B*n, Hkv, 16]; seq_lens int32 [B].
    Returns (out, lse, plan)."""
    return _decode("msa_decode", q, kv, q_scale, k_scale, v_scale,
                   softmax_scale, topk, block_table, seq_lens, n,
                   max_seqlen_k, workspace, out, lse, want_lse, stream)


def msa_decode_nvfp4(q, kv4, q_scale, k_scale, v_scale, softmax_scale, topk,
                     block_table, seq_lens, n, max_seqlen_k, workspace=None,
                     out=None, lse=None, want_lse=True, stream=None):
    """msa_decode over an NVFP4 pool (kv4 as in msa_prefill_nvfp4; k_scale /
    v_scale the global scales).  Returns (out, lse, plan)."""
    return _decode("msa_decode_nvfp4", q, kv4, q_scale, k_scale, v_scale,
                   softmax_scale, topk, block_table, seq_lens, n,
                   max_seqlen_k, workspace, out, lse, want_lse, stream)


def _decode(name, q, kv, q_scale, k_scale, v_scale, softmax_scale, topk,
            block_table, seq_lens, n, max_seqlen_k, workspace, out, lse,
            want_lse, stream):
    fp4 = name.endswith("nvfp4")
    B, Hq, Hkv = _decode_shapes(q, kv, topk, seq_lens, n, fp4, out, lse)
    _need(q, "q", _E4M3)
    _need(topk, "topk", (torch.int32,))
    _need(block_table, "block_table", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    _need_kv(kv, Hkv, fp4)
    need = decode_workspace_bytes(B, n, Hq, Hkv, max_seqlen_k)
    ws = _workspace(need, q.device, workspace)
    if out is None:
        out = torch.empty((B * n, Hq, HEAD_DIM), dtype=torch.bfloat16,
                          device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B * n, Hq), dtype=torch.float32, device=q.device)
    _need(out, "out", (torch.bfloat16,))
    if lse is not None:
        _need(lse, "lse", (torch.float32,))
    bt_stride = int(block_table.shape[1]) if block_table.dim() == 2 else 1
    st = MsaPlanStruct()
    _check(getattr(load(), name)(_ptr(_bytes(q)), _ptr(_bytes(kv)),
                                 int(kv.shape[0]), float(q_scale),
                                 float(k_scale), float(v_scale),
                                 float(softmax_scale), _ptr(topk),
                                 _ptr(block_table), bt_stride, _ptr(seq_lens),
                                 B, int(n), Hq, Hkv, int(max_seqlen_k),
                                 _ptr(ws), need, _ptr(out), _ptr(lse),
                                 ctypes.byref(st), _stream(stream)), name)
    return out, lse, Plan(st, ws, (topk, seq_lens, block_table))


def msa_decode_noalloc(q, kv, q_scale, k_scale, v_scale, softmax_scale,
                       topk, block_table, seq_lens, n, max_seqlen_k, out, lse,
                       stream=None):
    """msa_decode with the library's fixed device scratch instead of a
    workspace: for callers that cannot allocate device memory.  out and lse
    are the caller's; nothing is allocated here or in the library call.  The
    same shape checks as msa_decode run first, since the library sees only
    pointers and could not catch a mis-shaped pool or output."""
    if out is None:
        raise MsaError("out is required")
    B, Hq, Hkv = _decode_shapes(q, kv, topk, seq_lens, n, False, out, lse)
    _need(q, "q", _E4M3)
    _need(kv, "kv", _E4M3)
    _need(topk, "topk", (torch.int32,))
    _need(block_table, "block_table", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    _need(out, "out", (torch.bfloat16,))
    if lse is not None:
        _need(lse, "lse", (torch.float32,))
    bt_stride = int(block_table.shape[1]) if block_table.dim() == 2 else 1
    _check(load().msa_decode_noalloc(
        _ptr(_bytes(q)), _ptr(_bytes(kv)), int(kv.shape[0]), float(q_scale),
        float(k_scale), float(v_scale), float(softmax_scale), _ptr(topk),
        _ptr(block_table), bt_stride, _ptr(seq_lens), B, int(n), Hq, Hkv,
        int(max_seqlen_k), _ptr(out), _ptr(lse), _stream(stream)),
        "msa_decode_noalloc")
    return out, lse


def run_workload(w, stream=None):
    """Plan + prefill for a ``workloads.Workload`` already on the GPU;
    returns (out, lse, plan)."""
    plan = msa_plan(w.topk, w.cu_q, w.cu_k, w.block_table, w.num_pages, w.Hq,
                    w.total_rows, w.max_seqlen_q, w.max_seqlen_k,
                    stream=stream)
    if getattr(w, "q16", None) is not None:
        out, lse = msa_prefill_bf16q(w.q16, w.kv, w.q_scale, w.k_scale,
                                     w.v_scale, w.softmax_scale,
                                     w.block_table, plan, stream=stream)
    elif getattr(w, "kv4", None) is not None:
        out, lse = msa_prefill_nvfp4(w.q, w.kv4, w.q_scale, w.k_scale,
                                     w.v_scale, w.softmax_scale,
                                     w.block_table, plan, stream=stream)
    else:
        out, lse = msa_prefill(w.q, w.kv, w.q_scale, w.k_scale, w.v_scale,
                               w.softmax_scale, w.block_table, plan,
                               stream=stream)
    return out, lse, plan
