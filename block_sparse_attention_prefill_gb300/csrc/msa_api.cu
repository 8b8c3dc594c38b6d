// The C ABI of libmsa (declared in include/msa.h): host-side argument
// checks, workspace layout and the launch sequence of each call.  Nothing
// here allocates device memory or synchronises, except msa_read_status /
// msa_read_counters, which are documented to synchronise.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace msa {

namespace {
std::atomic<uint64_t> g_test_wait_ns{0};
}  // namespace

uint64_t pipeline_wait_limit_ns() {
  const uint64_t t = g_test_wait_ns.load(std::memory_order_relaxed);
  return t ? t : kWaitLimitNs;
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess || n <= 0)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

constexpr size_t kAlign = 256;
constexpr int64_t kI32Max = 2147483647;
constexpr int64_t kFp4PageBytes = MSA_NVFP4_PAGE_HEAD_BYTES;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Carves one workspace into 256-byte aligned pieces (or just measures).
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(int64_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = align_up(off + (size_t)count * sizeof(T));
    return p;
  }
};

struct PlanShape {
  int64_t B, T, Hq, Hkv, R, max_q, G, C, W, rows, ntiles, max_nnz, max_work;
};

int plan_shape(int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t R,
               int64_t max_q, PlanShape* s) {
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || R < 0 || max_q < 0)
    return MSA_ERR_SHAPE;
  if (Hq % Hkv != 0) return MSA_ERR_UNSUPPORTED;
  const int64_t G = Hq / Hkv;
  if (G < 1 || G > kTileM || Hkv > 127) return MSA_ERR_UNSUPPORTED;
  s->B = B;
  s->T = T;
  s->Hq = Hq;
  s->Hkv = Hkv;
  s->R = R;
  s->max_q = max_q;
  s->G = G;
  s->C = kTileM / G;
  s->W = 4 * ceil_div(max_q, 128);  // 32-bit words, a multiple of 4
  s->rows = Hkv * R;
  s->ntiles = ceil_div(s->rows, plan_tile_rows(s->rows, s->W));
  s->max_nnz = T * Hkv * kTopK;
  s->max_work = ceil_div(s->max_nnz, s->C) + std::min(s->rows, s->max_nnz);
  // every index the kernels form must fit in int32
  if (s->rows >= kI32Max || s->max_nnz >= kI32Max || s->max_work >= kI32Max ||
      T * Hq >= kI32Max / kTopK || B >= kI32Max / 2 ||
      (double)s->rows * (double)s->W * 4.0 > 9.0e15)
    return MSA_ERR_SHAPE;
  return MSA_OK;
}

// One work record: an int4 header plus one int4 per token of the chunk.
int64_t record_bytes(const PlanShape& s) { return 16 * (1 + s.C); }

// Lays out the plan workspace; with base == nullptr only the size counts.
size_t plan_layout(const PlanShape& s, void* base, msa_plan_t* pl) {
  Carver c(base);
  int32_t* req_off = c.take<int32_t>(s.B + 1);
  uint32_t* bitmap = c.take<uint32_t>(s.rows * s.W);
  int32_t* word_pre = c.take<int32_t>(s.rows * s.W);
  int32_t* row_cnt = c.take<int32_t>(s.rows);
  int32_t* row_loc = c.take<int32_t>(2 * s.rows);
  uint64_t* tile_state = c.take<uint64_t>(s.ntiles);
  int32_t* row_ptr = c.take<int32_t>(s.rows + 1);
  int32_t* q_idx = c.take<int32_t>(s.max_nnz);
  uint8_t* slot = c.take<uint8_t>(s.max_nnz);
  int32_t* work = c.take<int32_t>(4 * s.max_work);
  char* records = c.take<char>(s.max_work * record_bytes(s));
  int32_t* counters = c.take<int32_t>(4);
  uint16_t* slot_mask = c.take<uint16_t>(s.T * s.Hkv);
  uint32_t* status = c.take<uint32_t>(1);
  if (pl) {
    pl->req_off = req_off;
    pl->bitmap = bitmap;
    pl->word_pre = word_pre;
    pl->row_cnt = row_cnt;
    pl->row_loc = row_loc;
    pl->tile_state = tile_state;
    pl->records = records;
    pl->record_bytes = record_bytes(s);
    pl->row_ptr = row_ptr;
    pl->q_idx = q_idx;
    pl->slot = slot;
    pl->work = work;
    pl->counters = counters;
    pl->slot_mask = slot_mask;
    pl->status = status;
  }
  return c.off;
}

struct PartialBufs {
  uint8_t* o = nullptr;
  uint8_t* big = nullptr;
  float* lse = nullptr;
  float* vscale = nullptr;
};

// The prefill workspace: v_scale, then per (token, query head, top-k slot)
// a 128-byte E4M3 partial row, its lse, and a 256-byte bf16 overflow row
// (written only for halves of large magnitude).
size_t prefill_layout(int64_t T, int64_t Hq, void* base, PartialBufs* b) {
  Carver c(base);
  float* vs = c.take<float>(1);
  uint8_t* po = c.take<uint8_t>(T * Hq * kTopK * kD);
  float* pl = c.take<float>(T * Hq * kTopK);
  uint8_t* pb = c.take<uint8_t>(T * Hq * kTopK * 2 * kD);
  if (b) {
    b->o = po;
    b->big = pb;
    b->lse = pl;
    b->vscale = vs;
  }
  return c.off;
}

bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

// topk_hkv / h_begin: the KV heads of topk's layout and the first of this
// call's Hkv among them (a head shard; topk_hkv == Hkv, h_begin == 0 else).
int plan_impl(const int32_t* topk, const int32_t* cu_q, const int32_t* cu_k,
              const int32_t* block_table, int64_t bt_stride, int64_t num_pages,
              int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t R,
              int64_t max_q, int64_t max_k, void* ws, size_t ws_bytes,
              msa_plan_t* plan, cudaStream_t stream, int64_t topk_hkv = -1,
              int64_t h_begin = 0) {
  if (!plan) return MSA_ERR_NULL;
  PlanShape s;
  int rc = plan_shape(B, T, Hq, Hkv, R, max_q, &s);
  if (rc) return rc;
  if (topk_hkv < 0) topk_hkv = Hkv;
  if (h_begin < 0 || h_begin + Hkv > topk_hkv || topk_hkv > 127 ||
      T * topk_hkv >= kI32Max / kTopK)
    return MSA_ERR_SHAPE;
  if (max_k < 0 || max_k > kI32Max || num_pages < 0 || bt_stride < 0 ||
      max_q > max_k)
    return MSA_ERR_SHAPE;
  if (ceil_div(max_k, kPage) > (1 << 24)) return MSA_ERR_SHAPE;
  if (!cu_q || !cu_k) return MSA_ERR_NULL;
  if (T > 0 && (!topk || !block_table)) return MSA_ERR_NULL;
  if (B > 0 && R > 0 && bt_stride < 1) return MSA_ERR_SHAPE;
  // a request of max_k keys has ceil(max_k / 128) logical pages: its
  // block_table row must hold them
  if (B > 0 && bt_stride < ceil_div(max_k, kPage)) return MSA_ERR_SHAPE;
  if (!aligned(topk, 4) || !aligned(cu_q, 4) || !aligned(cu_k, 4) ||
      !aligned(block_table, 4))
    return MSA_ERR_ALIGN;
  const size_t need = plan_layout(s, nullptr, nullptr);
  if (!ws || ws_bytes < need) return MSA_ERR_WORKSPACE;
  if (!aligned(ws, kAlign)) return MSA_ERR_ALIGN;
  std::memset(plan, 0, sizeof(*plan));
  plan->B = B;
  plan->T = T;
  plan->Hq = Hq;
  plan->Hkv = Hkv;
  plan->total_rows = R;
  plan->max_seqlen_q = max_q;
  plan->max_seqlen_k = max_k;
  plan->num_pages = num_pages;
  plan->bt_stride = bt_stride;
  plan->bitmap_words = s.W;
  plan->chunk_tokens = s.C;
  plan->max_nnz = s.max_nnz;
  plan->max_work = s.max_work;
  plan->rows = s.rows;
  plan->cu_seqlens_q = cu_q;
  plan->cu_seqlens_k = cu_k;
  plan_layout(s, ws, plan);
  return cuda_rc(launch_plan(*plan, topk, block_table, stream, (int)topk_hkv, (int)h_begin));
}

int attention_impl(const uint8_t* q, const uint8_t* kv, int64_t num_pages,
                   float q_scale, float k_scale, float v_scale,
                   float softmax_scale, const int32_t* block_table,
                   int64_t bt_stride, const msa_plan_t* plan, void* ws,
                   size_t ws_bytes, cudaStream_t stream,
                   int kv_format = MSA_KV_E4M3, bool q_bf16 = false) {
  if (!plan) return MSA_ERR_NULL;
  const int64_t T = plan->T, Hq = plan->Hq;
  if (T == 0) return MSA_OK;
  if (!q || !kv || !block_table) return MSA_ERR_NULL;
  if (num_pages != plan->num_pages || bt_stride != plan->bt_stride)
    return MSA_ERR_SHAPE;
  if (num_pages * plan->Hkv * kPage >= kI32Max) return MSA_ERR_SHAPE;
  if (!(q_scale > 0.f) || !(k_scale > 0.f) || !(v_scale > 0.f) ||
      !(softmax_scale > 0.f) || !std::isfinite(q_scale * k_scale * softmax_scale))
    return MSA_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(kv, 16)) return MSA_ERR_ALIGN;
  const size_t need = prefill_layout(T, Hq, nullptr, nullptr);
  if (!ws || ws_bytes < need) return MSA_ERR_WORKSPACE;
  if (!aligned(ws, kAlign)) return MSA_ERR_ALIGN;
  AttnArgs a;
  a.q = q;
  a.kv = kv;
  a.num_pages = num_pages;
  a.score_log2 = (float)((double)q_scale * (double)k_scale *
                         (double)softmax_scale * 1.4426950408889634074);
  a.v_scale = v_scale;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.plan = plan;
  a.kv_format = kv_format;
  a.q_bf16 = q_bf16 ? 1 : 0;
  PartialBufs pb;
  prefill_layout(T, Hq, ws, &pb);
  a.part_o = pb.o;
  a.part_big = pb.big;
  a.part_lse = pb.lse;
  a.part_vscale = pb.vscale;
  if (num_pages == 0) return MSA_OK;
  return cuda_rc(launch_attention(a, stream));
}

int prefill_combine_impl(const msa_plan_t* plan, void* ws, size_t ws_bytes,
                         uint16_t* out, float* lse, cudaStream_t stream) {
  if (!plan) return MSA_ERR_NULL;
  const int64_t T = plan->T, Hq = plan->Hq;
  if (T == 0) return MSA_OK;
  if (!out) return MSA_ERR_NULL;
  if (!aligned(out, 8) || !aligned(lse, 4)) return MSA_ERR_ALIGN;
  const size_t need = prefill_layout(T, Hq, nullptr, nullptr);
  if (!ws || ws_bytes < need) return MSA_ERR_WORKSPACE;
  if (!aligned(ws, kAlign)) return MSA_ERR_ALIGN;
  PartialBufs pb;
  prefill_layout(T, Hq, ws, &pb);
  return cuda_rc(launch_combine_attn(pb.o, pb.big, pb.lse, pb.vscale, plan->slot_mask,
                                     Hq / plan->Hkv, T * Hq, out, lse, stream));
}

int prefill_impl(const uint8_t* q, const uint8_t* kv, int64_t num_pages,
                 float q_scale, float k_scale, float v_scale,
                 float softmax_scale, const int32_t* block_table,
                 int64_t bt_stride, const msa_plan_t* plan, void* ws,
                 size_t ws_bytes, uint16_t* out, float* lse,
                 cudaStream_t stream, int kv_format = MSA_KV_E4M3,
                 bool q_bf16 = false) {
  if (!plan) return MSA_ERR_NULL;
  if (plan->T == 0) return MSA_OK;
  if (!out) return MSA_ERR_NULL;
  if (!aligned(out, 8) || !aligned(lse, 4)) return MSA_ERR_ALIGN;
  int rc = attention_impl(q, kv, num_pages, q_scale, k_scale, v_scale,
                          softmax_scale, block_table, bt_stride, plan, ws,
                          ws_bytes, stream, kv_format, q_bf16);
  if (rc) return rc;
  return prefill_combine_impl(plan, ws, ws_bytes, out, lse, stream);
}

struct DecodeLayout {
  int64_t R;
  size_t cu_bytes, plan_bytes, prefill_bytes, total;
};

int decode_layout(int64_t B, int64_t n, int64_t Hq, int64_t Hkv,
                  int64_t max_k, DecodeLayout* d) {
  if (B < 0 || n < 1 || n > 8 || max_k < n || max_k > kI32Max)
    return MSA_ERR_SHAPE;
  if (B > kI32Max / 8) return MSA_ERR_SHAPE;
  d->R = B * ceil_div(max_k, kPage);
  PlanShape s;
  int rc = plan_shape(B, B * n, Hq, Hkv, d->R, n, &s);
  if (rc) return rc;
  d->cu_bytes = align_up(2 * (size_t)(B + 1) * sizeof(int32_t));
  d->plan_bytes = plan_layout(s, nullptr, nullptr);
  d->prefill_bytes = prefill_layout(B * n, Hq, nullptr, nullptr);
  d->total = d->cu_bytes + d->plan_bytes + d->prefill_bytes;
  return MSA_OK;
}

int decode_impl(const uint8_t* q, const uint8_t* kv, int64_t num_pages,
                float q_scale, float k_scale, float v_scale,
                float softmax_scale, const int32_t* topk,
                const int32_t* block_table, int64_t bt_stride,
                const int32_t* seq_lens, int64_t B, int64_t n, int64_t Hq,
                int64_t Hkv, int64_t max_seqlen_k, void* workspace,
                size_t workspace_bytes, uint16_t* out, float* lse,
                msa_plan_t* plan_out, cudaStream_t st, int kv_format) {
  DecodeLayout d;
  int rc = decode_layout(B, n, Hq, Hkv, max_seqlen_k, &d);
  if (rc) return rc;
  if (B == 0) return MSA_OK;
  if (!seq_lens) return MSA_ERR_NULL;
  if (!workspace || workspace_bytes < d.total) return MSA_ERR_WORKSPACE;
  if (!aligned(workspace, kAlign)) return MSA_ERR_ALIGN;
  char* ws = static_cast<char*>(workspace);
  int32_t* cu_q = reinterpret_cast<int32_t*>(ws);
  int32_t* cu_k = cu_q + (B + 1);
  msa_plan_t local;
  msa_plan_t* plan = plan_out ? plan_out : &local;
  // validate everything the plan checks before launching anything
  PlanShape s;
  rc = plan_shape(B, B * n, Hq, Hkv, d.R, n, &s);
  if (rc) return rc;
  if (!q || !kv || !out || !topk || !block_table) return MSA_ERR_NULL;
  if (bt_stride < 1 || bt_stride < ceil_div(max_seqlen_k, kPage) || num_pages < 0 ||
      num_pages * Hkv * kPage >= kI32Max)
    return MSA_ERR_SHAPE;
  if (!(q_scale > 0.f) || !(k_scale > 0.f) || !(v_scale > 0.f) ||
      !(softmax_scale > 0.f))
    return MSA_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 8) ||
      !aligned(lse, 4) || !aligned(topk, 4) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4))
    return MSA_ERR_ALIGN;
  if (launch_decode_seqlens(seq_lens, B, n, cu_q, cu_k, st) != cudaSuccess)
    return MSA_ERR_CUDA;
  rc = plan_impl(topk, cu_q, cu_k, block_table, bt_stride, num_pages, B, B * n,
                 Hq, Hkv, d.R, n, max_seqlen_k, ws + d.cu_bytes, d.plan_bytes,
                 plan, st);
  if (rc) return rc;
  return prefill_impl(q, kv, num_pages, q_scale, k_scale, v_scale,
                      softmax_scale, block_table, bt_stride, plan,
                      ws + d.cu_bytes + d.plan_bytes, d.prefill_bytes, out,
                      lse, st, kv_format);
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" {

int msa_version(void) { return 100; }

const char* msa_status_string(int code) {
  switch (code) {
    case MSA_OK: return "ok";
    case MSA_ERR_SHAPE: return "a size, count or stride is out of range";
    case MSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MSA_ERR_ALIGN: return "pointer not aligned as required";
    case MSA_ERR_WORKSPACE: return "workspace missing or too small";
    case MSA_ERR_CUDA: return "a CUDA call failed";
    case MSA_ERR_NULL: return "a required pointer is NULL";
    case MSA_ERR_TOO_LARGE:
      return "problem needs more scratch than msa_decode_noalloc's fixed array";
    case MSA_ERR_BUSY:
      return "msa_decode_noalloc is already being called from another thread";
    default: return "unknown status";
  }
}

int msa_plan_workspace_bytes(int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                             int64_t total_rows, int64_t max_seqlen_q,
                             size_t* bytes) {
  if (!bytes) return MSA_ERR_NULL;
  PlanShape s;
  int rc = plan_shape(B, T, Hq, Hkv, total_rows, max_seqlen_q, &s);
  if (rc) return rc;
  *bytes = plan_layout(s, nullptr, nullptr);
  return MSA_OK;
}

int msa_plan(const int32_t* topk, const int32_t* cu_seqlens_q,
             const int32_t* cu_seqlens_k, const int32_t* block_table,
             int64_t bt_stride, int64_t num_pages, int64_t B, int64_t T,
             int64_t Hq, int64_t Hkv, int64_t total_rows,
             int64_t max_seqlen_q, int64_t max_seqlen_k, void* workspace,
             size_t workspace_bytes, msa_plan_t* plan, void* stream) {
  return plan_impl(topk, cu_seqlens_q, cu_seqlens_k, block_table, bt_stride,
                   num_pages, B, T, Hq, Hkv, total_rows, max_seqlen_q,
                   max_seqlen_k, workspace, workspace_bytes, plan,
                   static_cast<cudaStream_t>(stream));
}

int msa_plan_heads(const int32_t* topk, int64_t topk_hkv, int64_t h_begin,
                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                   const int32_t* block_table, int64_t bt_stride, int64_t num_pages,
                   int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t total_rows,
                   int64_t max_seqlen_q, int64_t max_seqlen_k, void* workspace,
                   size_t workspace_bytes, msa_plan_t* plan, void* stream) {
  return plan_impl(topk, cu_seqlens_q, cu_seqlens_k, block_table, bt_stride,
                   num_pages, B, T, Hq, Hkv, total_rows, max_seqlen_q,
                   max_seqlen_k, workspace, workspace_bytes, plan,
                   static_cast<cudaStream_t>(stream), topk_hkv, h_begin);
}

int msa_prefill_workspace_bytes(int64_t T, int64_t Hq, size_t* bytes) {
  if (!bytes) return MSA_ERR_NULL;
  if (T < 0 || Hq <= 0 || T * Hq >= kI32Max / kTopK) return MSA_ERR_SHAPE;
  *bytes = prefill_layout(T, Hq, nullptr, nullptr);
  return MSA_OK;
}

int msa_prefill(const uint8_t* q, const uint8_t* kv, int64_t num_pages,
                float q_scale, float k_scale, float v_scale,
                float softmax_scale, const int32_t* block_table,
                int64_t bt_stride, const msa_plan_t* plan, void* workspace,
                size_t workspace_bytes, uint16_t* out, float* lse,
                void* stream) {
  return prefill_impl(q, kv, num_pages, q_scale, k_scale, v_scale,
                      softmax_scale, block_table, bt_stride, plan, workspace,
                      workspace_bytes, out, lse,
                      static_cast<cudaStream_t>(stream));
}

int msa_prefill_nvfp4(const uint8_t* q, const uint8_t* kv4, int64_t num_pages,
                      float q_scale, float k_scale, float v_scale,
                      float softmax_scale, const int32_t* block_table,
                      int64_t bt_stride, const msa_plan_t* plan,
                      void* workspace, size_t workspace_bytes, uint16_t* out,
                      float* lse, void* stream) {
  return prefill_impl(q, kv4, num_pages, q_scale, k_scale, v_scale,
                      softmax_scale, block_table, bt_stride, plan, workspace,
                      workspace_bytes, out, lse,
                      static_cast<cudaStream_t>(stream), MSA_KV_NVFP4);
}

int msa_nvfp4_to_e4m3(const uint8_t* kv4, int64_t page_heads, uint8_t* kv8,
                      void* stream) {
  if (page_heads < 0 || page_heads > (int64_t(1) << 40) / kFp4PageBytes)
    return MSA_ERR_SHAPE;
  if (page_heads == 0) return MSA_OK;
  if (!kv4 || !kv8) return MSA_ERR_NULL;
  if (!aligned(kv4, 16) || !aligned(kv8, 16)) return MSA_ERR_ALIGN;
  return cuda_rc(launch_nvfp4_to_e4m3(kv4, page_heads, kv8,
                                      static_cast<cudaStream_t>(stream)));
}

int msa_prefill_attention(const uint8_t* q, const uint8_t* kv,
                          int64_t num_pages, float q_scale, float k_scale,
                          float v_scale, float softmax_scale,
                          const int32_t* block_table, int64_t bt_stride,
                          const msa_plan_t* plan, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return attention_impl(q, kv, num_pages, q_scale, k_scale, v_scale,
                        softmax_scale, block_table, bt_stride, plan, workspace,
                        workspace_bytes, static_cast<cudaStream_t>(stream));
}

int msa_prefill_attention_nvfp4(const uint8_t* q, const uint8_t* kv4,
                                int64_t num_pages, float q_scale, float k_scale,
                                float v_scale, float softmax_scale,
                                const int32_t* block_table, int64_t bt_stride,
                                const msa_plan_t* plan, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return attention_impl(q, kv4, num_pages, q_scale, k_scale, v_scale,
                        softmax_scale, block_table, bt_stride, plan, workspace,
                        workspace_bytes, static_cast<cudaStream_t>(stream),
                        MSA_KV_NVFP4);
}

int msa_prefill_bf16q(const uint16_t* q16, const uint8_t* kv, int64_t num_pages,
                      float q_scale, float k_scale, float v_scale,
                      float softmax_scale, const int32_t* block_table,
                      int64_t bt_stride, const msa_plan_t* plan,
                      void* workspace, size_t workspace_bytes, uint16_t* out,
                      float* lse, void* stream) {
  return prefill_impl(reinterpret_cast<const uint8_t*>(q16), kv, num_pages, q_scale,
                      k_scale, v_scale, softmax_scale, block_table, bt_stride, plan,
                      workspace, workspace_bytes, out, lse,
                      static_cast<cudaStream_t>(stream), MSA_KV_E4M3, true);
}

int msa_prefill_attention_bf16q(const uint16_t* q16, const uint8_t* kv,
                                int64_t num_pages, float q_scale, float k_scale,
                                float v_scale, float softmax_scale,
                                const int32_t* block_table, int64_t bt_stride,
                                const msa_plan_t* plan, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return attention_impl(reinterpret_cast<const uint8_t*>(q16), kv, num_pages, q_scale,
                        k_scale, v_scale, softmax_scale, block_table, bt_stride, plan,
                        workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                        MSA_KV_E4M3, true);
}

int msa_prefill_combine(const msa_plan_t* plan, void* workspace,
                        size_t workspace_bytes, uint16_t* out, float* lse,
                        void* stream) {
  return prefill_combine_impl(plan, workspace, workspace_bytes, out, lse,
                              static_cast<cudaStream_t>(stream));
}

int msa_combine(const void* part_o, int part_dtype, const float* part_lse,
                int64_t rows, int64_t splits, uint16_t* out, float* lse_out,
                void* stream) {
  if (rows < 0 || splits < 1 || splits > 64 || rows >= kI32Max)
    return MSA_ERR_SHAPE;
  if (part_dtype != MSA_DTYPE_F32 && part_dtype != MSA_DTYPE_BF16)
    return MSA_ERR_UNSUPPORTED;
  if (rows == 0) return MSA_OK;
  if (!part_o || !part_lse || !out) return MSA_ERR_NULL;
  if (!aligned(part_o, part_dtype == MSA_DTYPE_F32 ? 16 : 8) ||
      !aligned(part_lse, 4) || !aligned(out, 8) || !aligned(lse_out, 4))
    return MSA_ERR_ALIGN;
  return cuda_rc(launch_combine(part_o, part_dtype, part_lse, rows,
                                splits, out, lse_out,
                                static_cast<cudaStream_t>(stream)));
}

int msa_decode_workspace_bytes(int64_t B, int64_t n, int64_t Hq, int64_t Hkv,
                               int64_t max_seqlen_k, size_t* bytes) {
  if (!bytes) return MSA_ERR_NULL;
  DecodeLayout d;
  int rc = decode_layout(B, n, Hq, Hkv, max_seqlen_k, &d);
  if (rc) return rc;
  *bytes = d.total;
  return MSA_OK;
}

int msa_decode(const uint8_t* q, const uint8_t* kv, int64_t num_pages,
               float q_scale, float k_scale, float v_scale,
               float softmax_scale, const int32_t* topk,
               const int32_t* block_table, int64_t bt_stride,
               const int32_t* seq_lens, int64_t B, int64_t n, int64_t Hq,
               int64_t Hkv, int64_t max_seqlen_k, void* workspace,
               size_t workspace_bytes, uint16_t* out, float* lse,
               msa_plan_t* plan_out, void* stream) {
  return decode_impl(q, kv, num_pages, q_scale, k_scale, v_scale,
                     softmax_scale, topk, block_table, bt_stride, seq_lens, B,
                     n, Hq, Hkv, max_seqlen_k, workspace, workspace_bytes, out,
                     lse, plan_out, static_cast<cudaStream_t>(stream),
                     MSA_KV_E4M3);
}

int msa_decode_nvfp4(const uint8_t* q, const uint8_t* kv4, int64_t num_pages,
                     float q_scale, float k_scale, float v_scale,
                     float softmax_scale, const int32_t* topk,
                     const int32_t* block_table, int64_t bt_stride,
                     const int32_t* seq_lens, int64_t B, int64_t n, int64_t Hq,
                     int64_t Hkv, int64_t max_seqlen_k, void* workspace,
                     size_t workspace_bytes, uint16_t* out, float* lse,
                     msa_plan_t* plan_out, void* stream) {
  return decode_impl(q, kv4, num_pages, q_scale, k_scale, v_scale,
                     softmax_scale, topk, block_table, bt_stride, seq_lens, B,
                     n, Hq, Hkv, max_seqlen_k, workspace, workspace_bytes, out,
                     lse, plan_out, static_cast<cudaStream_t>(stream),
                     MSA_KV_NVFP4);
}

}  // extern "C"

namespace {

// Scratch of msa_decode_noalloc: one fixed array on every GPU that loads this
// library, kept until the process exits.  Host code must not use its name
// as a device address; it asks the runtime for the address instead.
static __device__ __align__(256) unsigned char
    g_decode_scratch[MSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
std::atomic<int> g_noalloc_busy{0};

// The array's device address in the current device's context.  Outside
// stream capture it is looked up on every call (the runtime call is cheap
// once the module is loaded, and a fresh lookup stays right after a context
// is torn down and rebuilt); under capture, where the first lookup's module
// load must not happen, the address from this device's last call outside
// capture is used.
int decode_scratch(cudaStream_t stream, void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MSA_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return MSA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  } else if (g_scratch_ptr[dev] == nullptr) {
    return MSA_ERR_CUDA;  // no call outside capture on this device yet
  }
  *ptr = g_scratch_ptr[dev];
  return MSA_OK;
}

}  // namespace

extern "C" {

int msa_decode_noalloc(const uint8_t* q, const uint8_t* kv, int64_t num_pages,
                       float q_scale, float k_scale, float v_scale,
                       float softmax_scale, const int32_t* topk,
                       const int32_t* block_table, int64_t bt_stride,
                       const int32_t* seq_lens, int64_t B, int64_t n,
                       int64_t Hq, int64_t Hkv, int64_t max_seqlen_k,
                       uint16_t* out, float* lse, void* stream) {
  size_t need = 0;
  int rc = msa_decode_workspace_bytes(B, n, Hq, Hkv, max_seqlen_k, &need);
  if (rc) return rc;
  if (need > (size_t)MSA_NOALLOC_SCRATCH_BYTES) return MSA_ERR_TOO_LARGE;
  if (B == 0) return MSA_OK;
  // a second host thread entering while one is enqueueing would share the
  // array: refuse it instead of letting the two overwrite each other
  int expected = 0;
  if (!g_noalloc_busy.compare_exchange_strong(expected, 1)) return MSA_ERR_BUSY;
  void* scratch = nullptr;
  rc = decode_scratch(static_cast<cudaStream_t>(stream), &scratch);
  if (rc == MSA_OK)
    rc = msa_decode(q, kv, num_pages, q_scale, k_scale, v_scale, softmax_scale,
                    topk, block_table, bt_stride, seq_lens, B, n, Hq, Hkv,
                    max_seqlen_k, scratch, MSA_NOALLOC_SCRATCH_BYTES, out, lse,
                    nullptr, stream);
  g_noalloc_busy.store(0);
  return rc;
}

int msa_test_set_wait_limit_ns(uint64_t ns) {
  g_test_wait_ns.store(ns, std::memory_order_relaxed);
  return MSA_OK;
}

int msa_read_status(const msa_plan_t* plan, uint32_t* status) {
  if (!plan || !status || !plan->status) return MSA_ERR_NULL;
  return cuda_rc(cudaMemcpy(status, plan->status, sizeof(uint32_t),
                            cudaMemcpyDeviceToHost));
}

int msa_read_counters(const msa_plan_t* plan, int64_t* nnz,
                      int64_t* num_work) {
  if (!plan || !plan->counters) return MSA_ERR_NULL;
  int32_t c[4] = {0, 0, 0, 0};
  cudaError_t e =
      cudaMemcpy(c, plan->counters, sizeof(c), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  if (nnz) *nnz = c[0];
  if (num_work) *num_work = c[1];
  return MSA_OK;
}

}  // extern "C"
