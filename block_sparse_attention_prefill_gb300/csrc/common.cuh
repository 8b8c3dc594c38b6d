// Shared declarations of the libmsa translation units (plan, attention,
// combine, C ABI).  Shape constants follow the MSA pages: head dim 128,
// 128-token pages, top-16 pages per (token, KV head).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "msa.h"

namespace msa {

constexpr int kD = MSA_HEAD_DIM;      // head dim
constexpr int kPage = MSA_PAGE_SIZE;  // tokens per KV page
constexpr int kTopK = MSA_TOPK;       // pages per (token, KV head)
constexpr int kTileM = 128;           // MMA rows per work item (tokens x G)

// The plan's rows kernel: its threads, the lanes that share one row (the
// row's 16-byte vectors rounded up to a power of two, at most 16), and its
// tiles (CTAs).  A round is kRowThreads / lanes rows; a tile is the fewest
// whole rounds that keep the tile count within kMaxRowTiles, so the scatter
// kernel's CTAs can each scan all tiles' totals (one per thread).  A tile
// is worked in segments of at most kMaxTileRows rows.
constexpr int kRowThreads = 256;
constexpr int kMaxRowTiles = kRowThreads;
constexpr int kMaxTileRows = 512;  // a multiple of every round (16 .. 256 rows)
__host__ __device__ inline int plan_row_lane_shift(int64_t W) {
  const int64_t nv = W / 4;  // 16-byte vectors per row
  int s = 0;
  while (s < 4 && ((int64_t)1 << s) < nv) ++s;
  return s;
}
__host__ __device__ inline int64_t plan_tile_rows(int64_t rows, int64_t W) {
  const int64_t rp = kRowThreads >> plan_row_lane_shift(W);  // rows per round
  int64_t tr = (rows + kMaxRowTiles - 1) / kMaxRowTiles;
  tr = (tr + rp - 1) / rp * rp;
  return tr < rp ? rp : tr;
}

// A sparse plan: its membership bitmap holds at least 32 bytes per top-k
// entry, i.e. few tokens per selected page (long contexts, decode
// batches).  The plan's mark and scatter kernels and the attention kernel
// are tuned differently for sparse and dense plans (measured on GB300).
__host__ __device__ inline bool plan_is_sparse(int64_t rows, int64_t bitmap_words, int64_t T,
                                               int64_t Hkv) {
  return rows * bitmap_words * 4 >= 32 * T * Hkv * kTopK;
}

// Wall-time bound of every device-side wait (about a second).
constexpr uint32_t kWaitLimitNs = 1000000000u;

// The limit the attention kernel's pipeline waits use: kWaitLimitNs unless a
// test has set a shorter one (msa_test_set_wait_limit_ns).
uint64_t pipeline_wait_limit_ns();

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) {
  return (a + b - 1) / b;
}

// Launchers (each returns a cudaError_t from the launch).
// topk holds topk_hkv KV heads per token; the plan covers heads
// [h_begin, h_begin + plan.Hkv) of them.
cudaError_t launch_plan(const msa_plan_t& plan, const int32_t* topk,
                        const int32_t* block_table, cudaStream_t stream,
                        int topk_hkv, int h_begin);

// Split partials: per (token, query head, top-k slot) a 128-byte E4M3 row
// in V's code units, two halves of 64 columns.  A half with a value whose
// magnitude, in real units, is above kE4M3PartialLimit is kept in bf16 in
// the slot's 256-byte overflow row instead, and its E4M3 half holds the NaN
// code 0x7F in every byte as the marker.
constexpr float kE4M3PartialLimit = 2.0f;

struct AttnArgs {
  const uint8_t* q;
  const uint8_t* kv;
  int64_t num_pages;
  float score_log2;   // q_scale * k_scale * softmax_scale * log2(e)
  float v_scale;
  const int32_t* block_table;
  int64_t bt_stride;
  const msa_plan_t* plan;
  uint8_t* part_o;    // [T][Hq][16][128] E4M3: normalised partial outputs in
                      // V's code units (a convex combination of V codes)
  uint8_t* part_big;  // [T][Hq][16][128] bf16 overflow rows (see above)
  float* part_lse;    // [T][Hq][16]
  float* part_vscale; // one float: v_scale, left here for the combine
  int kv_format;      // MSA_KV_E4M3: kv is the E4M3 pool; MSA_KV_NVFP4: kv
                      // holds NVFP4 page-heads (nvfp4.cuh), dequantised to
                      // E4M3 in shared memory
  int q_bf16 = 0;     // 1: q is bf16 [T][Hq][128] (E4M3 pool only)
};

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream);
// The BF16-query kernel (attention_bf16q.cu); launch_attention calls it
// when a.q_bf16 is set.
cudaError_t launch_attention_bf16q(const AttnArgs& a, cudaStream_t stream);

// Combine over `splits` caller-given partials per row (bf16 or fp32 O,
// [rows][splits][128], lse [rows][splits], -inf marking an empty split).
cudaError_t launch_combine(const void* part_o, int part_dtype,
                           const float* part_lse, int64_t rows, int64_t splits,
                           uint16_t* out, float* lse, cudaStream_t stream);

// Combine of the attention kernel's partials: 16 slots per row, O in V's
// code units (each half E4M3, or bf16 in the overflow rows where the E4M3
// half holds the marker) scaled by *v_scale, the mask of row r is
// slot_mask[r / group] and empty slots are not read.
cudaError_t launch_combine_attn(const uint8_t* part_o, const uint8_t* part_big,
                                const float* part_lse, const float* v_scale,
                                const uint16_t* slot_mask, int64_t group,
                                int64_t rows, uint16_t* out, float* lse,
                                cudaStream_t stream);

cudaError_t launch_decode_seqlens(const int32_t* seq_lens, int64_t B,
                                  int64_t n, int32_t* cu_q, int32_t* cu_k,
                                  cudaStream_t stream);

// NVFP4 page-heads -> E4M3 pool [page_heads][128][256].
cudaError_t launch_nvfp4_to_e4m3(const uint8_t* kv4, int64_t page_heads,
                                 uint8_t* kv8, cudaStream_t stream);

int num_sms();

// Programmatic dependent launch.  A kernel launched with launch_pdl may
// start while the kernel before it in the stream is still running: it
// calls pdl_wait() before its first global-memory access, which returns
// once every earlier kernel of the stream has completed and its writes are
// visible.  pdl_trigger() lets the next kernel be scheduled early.  With
// no kernel in front (an event or a copy instead), pdl_wait() returns at
// once and the launch is ordinary.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                       size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace msa
