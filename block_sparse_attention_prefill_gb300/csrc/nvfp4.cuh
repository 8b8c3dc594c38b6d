// NVFP4 K/V pages read by an E4M3-query kernel (vLLM PR 60684, Details /
// "Kernel capability": with an E4M3 query, each NVFP4 code times its block
// scale is dequantised to E4M3, the K global scale goes on the scores and
// the V global scale into the combine; Details / "Numerics": the NVFP4
// kernel rounds K/V to E4M3).
//
// Page layout (the MSA backend over NVFP4 pages keeps, per KV head, a K slot
// and a V slot of packed data plus block scales; vLLM docs,
// MiniMaxM3SparseMSANvfp4Backend): for each (page, KV head), the K slot then
// the V slot; a slot is 128 tokens x 64 bytes of E2M1 codes (element 2i in
// the low nibble of byte i) followed by 128 tokens x 8 E4M3 block scales
// (scale b covers elements 16b .. 16b+15).
//
// One 16-element block -> 16 E4M3 bytes in element order, by table lookup:
// the E4M3 code of (E2M1 value x block scale) depends only on the scale
// code and the 3-bit magnitude, with the E2M1 sign flipping the result's.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace msa {

constexpr int kFp4Codes = 128 * 64;                 // code bytes per slot
constexpr int kFp4Slot = kFp4Codes + 128 * 8;       // one K or V slot
constexpr int kFp4PageHead = 2 * kFp4Slot;          // K slot + V slot

constexpr int kFp4LutBytes = 256 * 8;               // [scale code][8 magnitudes]

// Lookup table: entry (s, i) is the E4M3 code of E2M1 magnitude i (0, 0.5,
// 1, 1.5, 2, 3, 4, 6) times the E4M3 scale s.  The product is exact in fp32;
// the conversion rounds to nearest even and saturates at 448.  Built once
// per CTA by `nthreads` threads.
__device__ __forceinline__ void nvfp4_build_lut(uint8_t* lut, int tid, int nthreads) {
  for (int e = tid; e < kFp4LutBytes; e += nthreads) {
    const int scale = e >> 3, mag = e & 7;
    const __half2 m = __half2(__nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)mag, __NV_E2M1));
    const __half sc = __half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)scale, __NV_E4M3));
    const float x = __low2float(m) * __half2float(sc);
    lut[e] = (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
  }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four E2M1 codes in the low 16 bits of `codes` (the first in the low
// nibble; `mags` = the same with the sign bits cleared) -> four E4M3 bytes,
// the first in the low byte.  t0/t1: the block's eight magnitude codes.
// A byte permute looks up the magnitude index (bits 0-2 of each nibble); a
// second permute, whose nibbles keep their sign bit, gives 0xFF for a
// negative code (the sign-replicate mode of prmt on a 0x80 byte) and 0x80
// otherwise, and bit 0 of that byte, moved to bit 7, flips the sign of the
// looked-up code.  Flipping (rather than setting) the sign also gives the
// right sign of zero and of a negative scale.
__device__ __forceinline__ uint32_t fp4x4_lut(uint32_t codes, uint32_t mags,
                                              uint32_t t0, uint32_t t1) {
  const uint32_t mag = prmt(t0, t1, mags);
  const uint32_t neg = prmt(0x80808080u, 0x80808080u, codes);
  return mag ^ ((neg << 7) & 0x80808080u);
}

// codes: the block's 8 code bytes; scale: its E4M3 block-scale byte; lut:
// the table above.  Returns the 16 E4M3 bytes in element order.
__device__ __forceinline__ uint4 nvfp4_block_to_e4m3(uint2 codes, uint32_t scale,
                                                     const uint8_t* lut) {
  const uint2 t = *reinterpret_cast<const uint2*>(lut + scale * 8);
  const uint32_t m0 = codes.x & 0x77777777u, m1 = codes.y & 0x77777777u;
  return make_uint4(fp4x4_lut(codes.x, m0, t.x, t.y),
                    fp4x4_lut(codes.x >> 16, m0 >> 16, t.x, t.y),
                    fp4x4_lut(codes.y, m1, t.x, t.y),
                    fp4x4_lut(codes.y >> 16, m1 >> 16, t.x, t.y));
}

}  // namespace msa
