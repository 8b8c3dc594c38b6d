// NVFP4 page pool -> E4M3 page pool: the cache as an E4M3-query kernel reads
// it (vLLM PR 60684, Details).  The attention kernel does the same
// conversion in shared memory, with the same table and block routine
// (nvfp4.cuh); this
// kernel writes it out to global memory, for callers that stage pages and
// for checking the conversion bit for bit.
//
// One CTA per (page, KV head) at a time, grid-stride; 2048 blocks of 16
// elements per page-head (2 slots x 128 tokens x 8), one per thread and
// step.  Code loads are 8 contiguous bytes per thread, stores 16; the
// kernel is HBM-bound (18 KB read, 32 KB written per page-head).
#include "common.cuh"
#include "nvfp4.cuh"

namespace msa {
namespace {

constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads)
nvfp4_to_e4m3_kernel(const uint8_t* __restrict__ kv4, int64_t page_heads,
                     uint8_t* __restrict__ kv8) {
  __shared__ __align__(16) uint8_t lut[kFp4LutBytes];
  nvfp4_build_lut(lut, threadIdx.x, kStageThreads);
  __syncthreads();
  for (int64_t ph = blockIdx.x; ph < page_heads; ph += gridDim.x) {
    const uint8_t* src = kv4 + ph * kFp4PageHead;
    uint8_t* dst = kv8 + ph * (int64_t)(kPage * 2 * kD);
#pragma unroll 2
    for (int blk = threadIdx.x; blk < 2 * kPage * 8; blk += kStageThreads) {
      const int s = blk >> 10, rem = blk & 1023, t = rem >> 3, b = rem & 7;
      const uint8_t* slot = src + s * kFp4Slot;
      const uint2 codes = __ldg(reinterpret_cast<const uint2*>(slot + rem * 8));
      const uint32_t scale = __ldg(slot + kFp4Codes + rem);
      *reinterpret_cast<uint4*>(dst + t * (2 * kD) + s * kD + b * 16) =
          nvfp4_block_to_e4m3(codes, scale, lut);
    }
  }
}

}  // namespace

cudaError_t launch_nvfp4_to_e4m3(const uint8_t* kv4, int64_t page_heads,
                                 uint8_t* kv8, cudaStream_t stream) {
  if (page_heads <= 0) return cudaSuccess;
  const int64_t grid = std::min<int64_t>(page_heads, (int64_t)num_sms() * 8);
  nvfp4_to_e4m3_kernel<<<(unsigned)grid, kStageThreads, 0, stream>>>(kv4, page_heads, kv8);
  return cudaGetLastError();
}

}  // namespace msa
