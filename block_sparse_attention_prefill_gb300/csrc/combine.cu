// Split-KV combine: merge the per-slot partials of every (token, query head)
// by log-sum-exp and round to bf16.  (vLLM PR 60684, Performance: the
// per-layer call is build_k2q_csr + attention + combine; Validation: the
// E4M3 probabilities are rounded per split and the splits are merged.)
//
// For row r with filled slots j:  M = max lse_j,  sum = sum_j e^(lse_j - M),
// out = sum_j (e^(lse_j - M) / sum) * O_j,  lse = M + ln(sum).
// Two kernels: combine16_kernel merges the attention kernel's partials (16
// slots, E4M3 in V's code units, a half-warp per row); combine_kernel merges
// caller-given bf16 / fp32 partials for msa_combine (a warp per row, each
// lane owning 4 of the 128 columns).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 x = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&x.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&x.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
}

template <typename TIn, bool kMask>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
combine_kernel(const TIn* __restrict__ part_o, const float* __restrict__ part_lse,
               const uint16_t* __restrict__ slot_mask, int64_t group,
               int64_t rows, int S, uint16_t* __restrict__ out,
               float* __restrict__ lse_out) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (r >= rows) return;
  uint32_t mask = 0xffffffffu;
  if (kMask) mask = slot_mask[r / group];
  // split j = lane and j = lane + 32
  float l0 = -INFINITY, l1 = -INFINITY;
  if (lane < S && ((mask >> lane) & 1u)) l0 = part_lse[r * S + lane];
  if (!kMask && lane + 32 < S) l1 = part_lse[r * S + lane + 32];
  float M = fmaxf(l0, l1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  uint2* dst = reinterpret_cast<uint2*>(out + r * kD + lane * 4);
  if (M == -INFINITY) {
    *dst = make_uint2(0u, 0u);
    if (lse_out && lane == 0) lse_out[r] = -INFINITY;
    return;
  }
  const float w0 = (l0 == -INFINITY) ? 0.f : __expf(l0 - M);
  const float w1 = (l1 == -INFINITY) ? 0.f : __expf(l1 - M);
  float sum = w0 + w1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = 1.f / sum;
  const uint32_t live0 = __ballot_sync(0xffffffffu, w0 > 0.f);
  const uint32_t live1 = __ballot_sync(0xffffffffu, w1 > 0.f);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const TIn* base = part_o + r * (int64_t)S * kD + lane * 4;
  for (uint32_t bits = live0; bits; bits &= bits - 1) {
    const int j = __ffs(bits) - 1;
    const float wj = __shfl_sync(0xffffffffu, w0, j) * inv;
    float v[4];
    load4(base + (int64_t)j * kD, v);
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] = fmaf(wj, v[u], acc[u]);
  }
  for (uint32_t bits = live1; bits; bits &= bits - 1) {
    const int j = __ffs(bits) - 1;
    const float wj = __shfl_sync(0xffffffffu, w1, j) * inv;
    float v[4];
    load4(base + (int64_t)(j + 32) * kD, v);
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] = fmaf(wj, v[u], acc[u]);
  }
  __nv_bfloat162 a = __floats2bfloat162_rn(acc[0], acc[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(acc[2], acc[3]);
  *dst = make_uint2(*reinterpret_cast<uint32_t*>(&a),
                    *reinterpret_cast<uint32_t*>(&b));
  if (lse_out && lane == 0) lse_out[r] = M + __logf(sum);
}

// The attention path's combine: 16 slots per row, the slot mask of the
// row's (token, KV head) says which slots hold a partial.  Partial rows are
// E4M3 in V's code units (128 bytes); a half whose bytes are all the NaN
// code was kept in bf16 in the slot's overflow row instead (the attention
// kernel does that for halves of large magnitude).  The V scale is applied
// here, read from the device scalar the attention kernel left.  A
// half-warp per row, each lane owning 8 of the 128 columns: one 8-byte load
// per slot, all of a row's loads issued before any is used, and a 16-byte
// overflow load for a marked half.  The partials are read once here: they
// are evicted from L2 first.  With the weights normalised first, the sum is
// a convex combination of values within E4M3's range, accumulated in packed
// f16 (one conversion and one HFMA2 per pair of values).
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
combine16_kernel(const uint8_t* __restrict__ part_o,
                 const uint8_t* __restrict__ part_big,
                 const float* __restrict__ part_lse,
                 const float* __restrict__ v_scale_ptr,
                 const uint16_t* __restrict__ slot_mask, int64_t group,
                 int64_t rows, uint16_t* __restrict__ out,
                 float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;                 // lane within the half-warp
  const int64_t r = ((int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * 2 +
                    (lane >> 4);
  const bool live = r < rows;
  // The slot masks are the plan's, complete once the attention kernel has
  // passed its own wait, which is before it let this kernel launch: read
  // before this kernel's wait (through L2), which covers the partials.
  const uint32_t mask = live ? __ldcg(slot_mask + r / group) : 0u;
  pdl_wait();
  pdl_trigger();
  const uint64_t pol = l2_policy_evict_first();
  const uint8_t* base = part_o + r * (int64_t)kTopK * kD + sub * 8;
  uint2 v[kTopK];
#pragma unroll
  for (int j = 0; j < kTopK; ++j) {
    if ((mask >> j) & 1u)
      v[j] = ld_global_v2_hint(base + j * kD, pol);
    else
      v[j] = make_uint2(0u, 0u);
  }
  // lane `sub` of the half-warp holds slot sub's lse
  float l = -INFINITY;
  if ((mask >> sub) & 1u) l = ld_global_f32_hint(part_lse + r * kTopK + sub, pol);
  float M = l;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float wl = (l == -INFINITY) ? 0.f : __expf(l - M);
  float sum = wl;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  // normalised weights: the sums below stay convex combinations of the
  // partials, within +-448 (V's code units), so they are kept in packed
  // f16 (2^-11 relative per step, below the bf16 output's 2^-9)
  wl *= 1.f / sum;
  // every lane runs the loops below (their shuffles span the warp); rows
  // past the end or with no partial are written after them
  __half2 acc[4];  // columns (2u, 2u + 1) of this lane's 8
#pragma unroll
  for (int u = 0; u < 4; ++u) acc[u] = __float2half2_rn(0.f);
  uint32_t marked = 0;  // slots whose half (this lane's) is in the overflow rows
#pragma unroll
  for (int j = 0; j < kTopK; ++j) {
    const __half2 wj = __float2half2_rn(__shfl_sync(0xffffffffu, wl, (lane & 16) + j));
    // a marked half counts here as zeros (its NaN bytes must not reach the
    // sums); its bf16 values are added below
    const bool mk = v[j].x == 0x7F7F7F7Fu;
    marked |= (uint32_t)mk << j;
    const uint32_t w2[2] = {mk ? 0u : v[j].x, mk ? 0u : v[j].y};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
          (__nv_fp8x2_storage_t)(w2[u] & 0xFFFFu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
          (__nv_fp8x2_storage_t)(w2[u] >> 16), __NV_E4M3);
      acc[2 * u] = __hfma2(wj, *reinterpret_cast<const __half2*>(&lo), acc[2 * u]);
      acc[2 * u + 1] = __hfma2(wj, *reinterpret_cast<const __half2*>(&hi), acc[2 * u + 1]);
    }
  }
  // halves kept in bf16 (rare): this lane's 8 columns are 16 bytes of the
  // slot's overflow row
  // (the loop runs over the slots marked anywhere in the warp, so that every
  // lane takes part in the shuffle that fetches the slot's weight)
  const uint8_t* big = part_big + r * (int64_t)kTopK * (2 * kD) + sub * 16;
  marked &= mask;
  for (uint32_t bits = __reduce_or_sync(0xffffffffu, marked); bits; bits &= bits - 1) {
    const int j = __ffs(bits) - 1;
    const __half2 wj = __float2half2_rn(__shfl_sync(0xffffffffu, wl, (lane & 16) + j));
    if ((marked >> j) & 1u) {
      const uint4 b4 = ld_global_v4_hint(big + j * (2 * kD), pol);
      const uint32_t w4[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        acc[u] = __hfma2(wj,
                         __floats2half2_rn(__uint_as_float(w4[u] << 16),
                                           __uint_as_float(w4[u] & 0xFFFF0000u)),
                         acc[u]);
    }
  }
  if (!live) return;
  uint4* dst = reinterpret_cast<uint4*>(out + r * kD + sub * 8);
  if (M == -INFINITY) {
    *dst = make_uint4(0u, 0u, 0u, 0u);
    if (lse_out && sub == 0) lse_out[r] = -INFINITY;
    return;
  }
  const float vs = *v_scale_ptr;
  uint32_t o[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 a = __half22float2(acc[u]);
    __nv_bfloat162 h = __floats2bfloat162_rn(a.x * vs, a.y * vs);
    o[u] = *reinterpret_cast<uint32_t*>(&h);
  }
  *dst = make_uint4(o[0], o[1], o[2], o[3]);
  if (lse_out && sub == 0) lse_out[r] = M + __logf(sum);
}

__global__ void __launch_bounds__(1024)
decode_seqlens_kernel(const int32_t* seq_lens, int64_t B, int64_t n,
                      int32_t* cu_q, int32_t* cu_k) {
  pdl_wait();
  pdl_trigger();
  __shared__ int warp_sums[33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int carry = 0;
  for (int64_t base = 0; base < B; base += 1024) {
    const int64_t b = base + threadIdx.x;
    const int v = b < B ? seq_lens[b] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int s = warp_sums[lane];
      int si = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, si, o);
        if (lane >= o) si += x;
      }
      warp_sums[lane] = si - s;
      if (lane == 31) warp_sums[32] = si;
    }
    __syncthreads();
    if (b < B) {
      cu_k[b + 1] = carry + warp_sums[warp] + incl;
      cu_q[b + 1] = (int32_t)((b + 1) * n);
    }
    carry += warp_sums[32];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    cu_q[0] = 0;
    cu_k[0] = 0;
  }
}

}  // namespace

cudaError_t launch_combine(const void* part_o, int part_dtype,
                           const float* part_lse, int64_t rows, int64_t splits,
                           uint16_t* out, float* lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const dim3 grid((unsigned)ceil_div(rows, kWarpsPerBlock));
  const dim3 block(kWarpsPerBlock * 32);
  const uint16_t* no_mask = nullptr;
  const int64_t one = 1;
  const int S = (int)splits;
  if (part_dtype == MSA_DTYPE_BF16)
    return launch_pdl(combine_kernel<__nv_bfloat16, false>, grid, block, 0, stream,
                      static_cast<const __nv_bfloat16*>(part_o), part_lse, no_mask,
                      one, rows, S, out, lse);
  return launch_pdl(combine_kernel<float, false>, grid, block, 0, stream,
                    static_cast<const float*>(part_o), part_lse, no_mask, one, rows,
                    S, out, lse);
}

cudaError_t launch_combine_attn(const uint8_t* part_o, const uint8_t* part_big,
                                const float* part_lse, const float* v_scale,
                                const uint16_t* slot_mask, int64_t group,
                                int64_t rows, uint16_t* out, float* lse,
                                cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  return launch_pdl(combine16_kernel,
                    dim3((unsigned)ceil_div(rows, 2 * kWarpsPerBlock)),
                    dim3(kWarpsPerBlock * 32), 0, stream, part_o, part_big, part_lse,
                    v_scale, slot_mask, group, rows, out, lse);
}

cudaError_t launch_decode_seqlens(const int32_t* seq_lens, int64_t B,
                                  int64_t n, int32_t* cu_q, int32_t* cu_k,
                                  cudaStream_t stream) {
  return launch_pdl(decode_seqlens_kernel, dim3(1), dim3(1024), 0, stream, seq_lens, B, n,
                    cu_q, cu_k);
}

}  // namespace msa
