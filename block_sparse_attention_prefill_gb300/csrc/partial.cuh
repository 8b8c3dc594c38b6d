// Writing one split partial: the normalised O row of a (token, query head,
// top-k slot) in V's code units, as the combine kernel reads it.  Shared by
// the E4M3-query and the BF16-query attention kernels.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"

namespace msa {

// Two floats rounded to bf16 (nearest even) in one word, the first in the
// low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Four floats rounded to E4M3 (nearest even, saturating) in one word, the
// first in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// One 64-column half of a partial row: ra holds columns 0-31 of the half and
// rb columns 32-63 (fp32 bits, unnormalised), inv the row's 1 / l.
//
// The normalised row in V's code units is a convex combination of E4M3 V
// codes, so it stays within E4M3's range; word k holds columns 4k .. 4k+3
// of the half.  A half with a code above the limit that over4 encodes
// (magnitude kE4M3PartialLimit, 2.0 in real units) goes to the bf16
// overflow row instead (error at most 2^-9 of the value), and its E4M3 half
// is filled with the NaN code, which no partial produces (the conversion
// saturates), as the marker the combine looks for.  So the E4M3 rounding
// error of a partial stays at most 2^-4 * 2.0 = 0.125 absolute however large
// the output, and the common case moves 64 bytes a half.
//   d     the half's 64 bytes in the E4M3 partial row
//   big   the half's 128 bytes in the bf16 overflow row
//   over4 (0x7F - largest E4M3 magnitude code the half may keep) in each byte
__device__ __forceinline__ void store_partial_half(const uint32_t (&ra)[32],
                                                   const uint32_t (&rb)[32], float inv,
                                                   uint8_t* d, uint8_t* big, uint32_t over4,
                                                   uint64_t pol) {
  uint32_t o[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    o[k] = pack_e4m3x4(__uint_as_float(ra[4 * k]) * inv, __uint_as_float(ra[4 * k + 1]) * inv,
                       __uint_as_float(ra[4 * k + 2]) * inv,
                       __uint_as_float(ra[4 * k + 3]) * inv);
    o[8 + k] = pack_e4m3x4(__uint_as_float(rb[4 * k]) * inv, __uint_as_float(rb[4 * k + 1]) * inv,
                           __uint_as_float(rb[4 * k + 2]) * inv,
                           __uint_as_float(rb[4 * k + 3]) * inv);
  }
  // any magnitude byte above the limit: (b & 0x7F) + (0x7F - limit) carries
  // into bit 7 exactly when b & 0x7F exceeds the limit, and no byte carries
  // into the next (both terms are at most 0x7F)
  uint32_t over = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) over |= (o[k] & 0x7F7F7F7Fu) + over4;
  if (!(over & 0x80808080u)) {
    // 64 bytes as two whole 32-byte sectors
    st_global_v8_hint(d, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7], pol);
    st_global_v8_hint(d + 32, o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15], pol);
  } else {
    constexpr uint32_t kNaN4 = 0x7F7F7F7Fu;
    st_global_v8_hint(d, kNaN4, kNaN4, kNaN4, kNaN4, kNaN4, kNaN4, kNaN4, kNaN4, pol);
    st_global_v8_hint(d + 32, kNaN4, kNaN4, kNaN4, kNaN4, kNaN4, kNaN4, kNaN4, kNaN4, pol);
    // word k holds columns 2k, 2k+1; 128 bytes as four sectors
#pragma unroll
    for (int k = 0; k < 16; ++k)
      o[k] = pack_bf16x2(__uint_as_float(ra[2 * k]) * inv, __uint_as_float(ra[2 * k + 1]) * inv);
    st_global_v8_hint(big, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7], pol);
    st_global_v8_hint(big + 32, o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15], pol);
#pragma unroll
    for (int k = 0; k < 16; ++k)
      o[k] = pack_bf16x2(__uint_as_float(rb[2 * k]) * inv, __uint_as_float(rb[2 * k + 1]) * inv);
    st_global_v8_hint(big + 64, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7], pol);
    st_global_v8_hint(big + 96, o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15], pol);
  }
}

// (0x7F - c) in each byte, c the largest E4M3 magnitude code whose value
// (in V's code units) is at most kE4M3PartialLimit / v_scale; every code
// when that passes 448.
uint32_t partial_over4(float v_scale);

}  // namespace msa
