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

// Rows per CTA in the plan's fill kernel, and in its count kernel (a
// half-warp per row there).
constexpr int kPlanTile = 256;
constexpr int kCountTile = 16;

// Wall-time bound of every device-side wait (about a second).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) {
  return (a + b - 1) / b;
}

// Launchers (each returns a cudaError_t from the launch).
cudaError_t launch_plan(const msa_plan_t& plan, const int32_t* topk,
                        const int32_t* block_table, cudaStream_t stream);

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
  float* part_lse;    // [T][Hq][16]
  float* part_vscale; // one float: v_scale, left here for the combine
  int kv_format;      // MSA_KV_E4M3: kv is the E4M3 pool; MSA_KV_NVFP4: kv
                      // holds NVFP4 page-heads (nvfp4.cuh), dequantised to
                      // E4M3 in shared memory
};

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream);

// Combine over `splits` caller-given partials per row (bf16 or fp32 O,
// [rows][splits][128], lse [rows][splits], -inf marking an empty split).
cudaError_t launch_combine(const void* part_o, int part_dtype,
                           const float* part_lse, int64_t rows, int64_t splits,
                           uint16_t* out, float* lse, cudaStream_t stream);

// Combine of the attention kernel's partials: 16 slots per row, E4M3 O in
// V's code units scaled by *v_scale, the mask of row r is
// slot_mask[r / group] and empty slots are not read.
cudaError_t launch_combine_attn(const uint8_t* part_o, const float* part_lse,
                                const float* v_scale, const uint16_t* slot_mask,
                                int64_t group, int64_t rows, uint16_t* out,
                                float* lse, cudaStream_t stream);

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
