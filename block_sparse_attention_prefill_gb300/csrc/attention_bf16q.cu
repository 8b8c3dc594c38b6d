// Block-sparse attention with a BF16 query over the E4M3 page pool, for
// sm_103a: the K and V halves of each selected page are widened to bf16 in
// shared memory (exactly: every E4M3 value is a bf16 value), and QK and PV
// run as bf16 tensor-core MMAs (tcgen05, kind::f16) accumulating in tensor
// memory; the probabilities are rounded to bf16.  The work items, their
// records and the split partials (E4M3 in V's code units, bf16 overflow
// halves, fp32 lse) are those of the E4M3-query kernel, so the plan and the
// combine are shared.
//
// What it computes follows vLLM PR 60684 (Details / "Kernel capability":
// sparse_atten_func's BF16-Q x FP8-K/V mode stages K/V up to BF16 and runs
// BF16 MMAs; Performance: a BF16 query over the FP8 cache reaches the
// Blackwell port with BF16 MMAs) and the vLLM docs for sparse_attention_msa
// (MiniMaxM3SparseMSAImpl.forward: sparse_atten_func over the k2q CSR,
// causal=True, page_table=block_table).  The kernel design is this
// library's own.
//
// Three CTAs of four warps per SM, persistent; work items are dealt
// round-robin as in the E4M3-query kernel.  Per item, all 128 threads:
//   1. the record into shared memory; the Q rows (256 bytes each) by
//      cp.async into a 128 x 128 bf16 K-major tile (128-byte swizzle, two
//      64-column blocks);
//   2. the page-head's K codes, which each thread loaded into registers
//      during the previous item, widened into the K/V tile
//      [128 keys][128 dims] (same layout); the V codes are loaded now;
//   3. QK: 8 MMAs of K = 16 into S (TMEM columns 0-127);
//   4. the V codes widened into the same tile (K is dead once QK is done);
//      each thread takes its row of S (its TMEM lane), masks the keys after
//      its query, and writes P = 2^(s c - m c) in bf16 over its Q row;
//   5. PV: 8 MMAs into O, over the same TMEM columns as S (S is in
//      registers by then), V read MN-major; the next item's K codes are
//      loaded into registers while PV and the epilogue run;
//   6. each thread normalises its O row and writes the partial.
// The other two CTAs on the SM fill one CTA's waits.
#include <cuda.h>
#include <atomic>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "partial.cuh"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kThreadsB = 128;
constexpr int kCtasPerSm = 3;
constexpr int kBlockB = 128 * 128;          // 128 rows x 64 bf16 columns (16 KB)
constexpr int kOffKV = 0;                   // K, then V: bf16 [128 keys][128 dims]
constexpr int kOffQP = 2 * kBlockB;         // Q, then P: bf16 [128 rows][128]
constexpr int kOffRec = 4 * kBlockB;
constexpr int kOffBars = kOffRec + 16 * (1 + kTileM);
constexpr int kTmemColsB = 128;             // S, then O
constexpr int kChunks = kPage * 16 / kThreadsB;  // 8-code chunks of a half per thread
struct BarsB {
  uint64_t mma;       // QK (even phases) and PV (odd phases) completed
  uint64_t mma_done;  // every MMA completed, before the CTA exits
  uint32_t tmem_base;
  int abort;
};
constexpr int kSmemB = kOffBars + (int)sizeof(BarsB) + 1024;
static_assert(kOffBars % 8 == 0, "alignment");
// kCtasPerSm CTAs per SM: 228 KB of shared memory, 1 KB of it reserved per
// CTA, and 512 TMEM columns
static_assert(kCtasPerSm * (kSmemB + 1024) <= 233472, "the CTAs of an SM must fit");
static_assert(kCtasPerSm * kTmemColsB <= 512, "tensor memory of an SM");

struct ParamsB {
  const uint16_t* q16;   // bf16 [T][Hq][128]
  const uint8_t* kv;     // E4M3 pool, rows of 256 bytes (K | V)
  const int4* records;
  int rec_stride;        // int4 per record
  const int32_t* counters;
  uint8_t* part_o;
  uint8_t* part_big;
  float* part_vscale;
  float* part_lse;
  uint32_t e4m3_over4;
  uint32_t* status;
  int Hq, G;
  float score_log2;      // q_scale * k_scale * softmax_scale * log2(e)
  float v_scale;
  uint32_t wait_ns;
};

// Wait for the phase with the given parity, polling (no suspending wait)
// with a short sleep and a look at the clock each time, so that even a
// limit below one page load runs out; false on timeout or abort.
__device__ __forceinline__ bool poll_wait(uint64_t* bar, uint32_t parity,
                                          const volatile int* abort, uint32_t limit_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint32_t t0 = (uint32_t)global_timer_ns();
  for (;;) {
    __nanosleep(32);
    if (mbar_test(bar, parity)) return true;
    if (*abort || (uint32_t)global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Two E4M3 codes (low 16 bits) widened to two bf16 in one word, the first
// in the low half; exact, by way of f16.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu),
                                                   __NV_E4M3);
  const float2 f = __half22float2(__half2(h));
  return pack_bf16x2(f.x, f.y);
}

// A page-head is 128 token rows of 256 bytes, K in bytes 0-127 and V in
// 128-255.  Thread tid owns the 8-code chunks e = tid + 128 j (j < 16) of
// each half: chunk e is codes 8 (e % 16) .. +7 of token row e / 16, so a
// warp's loads cover two whole 128-byte half-rows.
__device__ __forceinline__ void load_codes(const uint8_t* page, int half, int tid,
                                           uint2 (&c)[kChunks]) {
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const int e = tid + j * kThreadsB;
    c[j] = ldg_nc_v2(page + (e >> 4) * (2 * kD) + half + (e & 15) * 8);
  }
}

// The chunks above widened into the bf16 tile [128 tokens][128 dims]: dims
// 0-63 in block 0, 64-127 in block 1, 128 bytes a row, 16-byte chunk c of
// row t at chunk c ^ (t & 7) (the 128-byte swizzle).  A warp's 16-byte
// stores cover whole rows of a block: no bank conflicts.
__device__ __forceinline__ void store_widened(const uint2 (&c)[kChunks], uint8_t* tile,
                                              int tid) {
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const int e = tid + j * kThreadsB, t = e >> 4, ch = e & 15;
    const uint4 w = make_uint4(e4m3x2_to_bf16x2(c[j].x), e4m3x2_to_bf16x2(c[j].x >> 16),
                               e4m3x2_to_bf16x2(c[j].y), e4m3x2_to_bf16x2(c[j].y >> 16));
    *reinterpret_cast<uint4*>(tile + (ch >> 3) * kBlockB + t * 128 +
                              (((ch & 7) ^ (t & 7)) << 4)) = w;
  }
}

// p = 2^(x * c + off) for 32 score columns starting at col0, rounded to
// bf16 and stored as four 16-byte chunks of the row's P (K-major bf16,
// 128-byte swizzle); adds the unrounded probabilities to l.  Masked
// columns hold -inf and give 0.
__device__ __forceinline__ void exp_store32(const uint32_t (&r)[32], int col0, float c,
                                            float off, uint8_t* prow, int row, float& l) {
  float lq[2] = {0.f, 0.f};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = ex2_approx(fmaf(__uint_as_float(r[q * 8 + 2 * k]), c, off));
      const float b = ex2_approx(fmaf(__uint_as_float(r[q * 8 + 2 * k + 1]), c, off));
      lq[0] += a;
      lq[1] += b;
      w[k] = pack_bf16x2(a, b);
    }
    const int ch = (col0 >> 3) + q;  // 8-column chunk 0 .. 15
    *reinterpret_cast<uint4*>(prow + (ch >> 3) * kBlockB + (((ch & 7) ^ (row & 7)) << 4)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  l += lq[0] + lq[1];
}

__device__ __forceinline__ void max_mask32(uint32_t (&r)[32], int col0, int kv_lim, float& m) {
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    if (col0 + e > kv_lim) r[e] = 0xFF800000u;  // -inf
    m = fmaxf(m, __uint_as_float(r[e]));
  }
}

__global__ void __launch_bounds__(kThreadsB, kCtasPerSm) attention_bf16q_kernel(const ParamsB p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BarsB* bars = reinterpret_cast<BarsB*>(smem + kOffBars);
  int4* srec = reinterpret_cast<int4*>(smem + kOffRec);
  uint8_t* kvt = smem + kOffKV;
  uint8_t* qp = smem + kOffQP;
  const int tid = threadIdx.x, warp = tid >> 5;

  // the plan's counters and records are written by the kernels before this
  // one in the stream
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && tid == 0) *p.part_vscale = p.v_scale;
  const int num_work = (*p.status & MSA_STATUS_TIMEOUT) ? 0 : p.counters[1];
  const int cnt = blockIdx.x < (unsigned)num_work
                      ? (num_work - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                      : 0;
  const int4* grec = p.records + (int64_t)blockIdx.x * p.rec_stride;
  const int64_t rec_step = (int64_t)gridDim.x * p.rec_stride;

  if (tid == 0) {
    mbar_init(&bars->mma, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(&bars->tmem_base, kTmemColsB);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const int row = tid;  // tile row = TMEM lane
  const uint64_t pol_keep = l2_policy_evict_last();

  // this thread's K code chunks, loaded one item ahead, and V code chunks,
  // loaded when the item starts (a page-head is the rows of 256 bytes from
  // the record's KV row)
  uint2 kc[kChunks], vc[kChunks];
  auto page_of = [&](int li) { return p.kv + (int64_t)grec[li * rec_step].x * (2 * kD); };
  if (cnt > 0) load_codes(page_of(0), 0, tid, kc);

  constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
  constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, true);
  bool failed = false;
  for (int li = 0; li < cnt; ++li) {
    const int4* rec = grec + li * rec_step;
    const int4 hdr = rec[0];
    const int n = hdr.y;
    load_codes(p.kv + (int64_t)hdr.x * (2 * kD), kD, tid, vc);
    for (int e = tid; e <= n; e += kThreadsB) srec[e] = rec[e];
    __syncthreads();

    // 1. Q rows: 16-byte chunk c of row lrow = (token i, head g)
    for (int e = tid; e < n * p.G * 16; e += kThreadsB) {
      const int lrow = e >> 4, c = e & 15;
      const int i = lrow / p.G, g = lrow - i * p.G;
      const uint16_t* src =
          p.q16 + ((int64_t)srec[1 + i].x * p.Hq + hdr.w + g) * kD + c * 8;
      cp_async_16(smem_u32(qp + (c >> 3) * kBlockB + lrow * 128 + (((c & 7) ^ (lrow & 7)) << 4)),
                  src);
    }
    cp_async_commit();

    // 2. K widened (its codes were loaded during the previous item)
    store_widened(kc, kvt, tid);
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // 3. QK: A = Q [128 rows][128 dims], B = K [128 keys][128 dims], both
    // K-major; K = 16 per MMA: 32 bytes into a 128-byte row, then the next
    // 64-column block
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (uint32_t)((kk >> 2) * kBlockB + (kk & 3) * 32);
        mma_f16(tmem, smem_desc_sw128(smem_u32(qp + off), 16, 1024),
                smem_desc_sw128(smem_u32(kvt + off), 16, 1024), idesc_qk, kk > 0);
      }
      mma_commit(&bars->mma);
    }
    bool ok = poll_wait(&bars->mma, 0, &bars->abort, p.wait_ns);
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();

    // 4. V widened over K; the row's softmax, P over the row's Q
    store_widened(vc, kvt, tid);
    const int i = row / p.G, g = row - i * p.G;
    const bool valid = i < n;
    const bool warp_valid = __any_sync(0xffffffffu, valid);
    int32_t prow = -1;
    int kv_lim = 127;
    if (valid) {
      const int4 tok = srec[1 + i];
      prow = (tok.x * p.Hq + hdr.w + g) * kTopK + tok.z;
      kv_lim = min(tok.y - hdr.z, 127);
    }
    float m2 = -INFINITY, l = 0.f;
    if (warp_valid) {
      // two passes over S in 32-column pieces (tensor memory is read twice
      // rather than holding the row's 128 scores in registers): the
      // maximum, then the probabilities
      float m = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + c * 32, r);
        tmem_wait_ld();
        max_mask32(r, c * 32, kv_lim, m);
      }
      m2 = m * p.score_log2;
      const float off = (m2 == -INFINITY) ? 0.f : -m2;
      uint8_t* prow_s = qp + row * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + c * 32, r);
        tmem_wait_ld();
        float unused = -INFINITY;
        max_mask32(r, c * 32, kv_lim, unused);
        exp_store32(r, c * 32, p.score_log2, off, prow_s, row, l);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // 5. PV into the S columns: A = P [128 rows][128 keys] K-major, B = V
    // [128 keys][128 dims] MN-major: 16 keys per MMA are 16 rows (2 KB)
    // further; the two 64-dim blocks are 16 KB apart (leading byte offset),
    // groups of 8 key rows 1 KB apart (stride byte offset)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a_off = (uint32_t)((kk >> 2) * kBlockB + (kk & 3) * 32);
        mma_f16(tmem, smem_desc_sw128(smem_u32(qp + a_off), 16, 1024),
                smem_desc_sw128(smem_u32(kvt + kk * 16 * 128), kBlockB, 1024), idesc_pv,
                kk > 0);
      }
      mma_commit(&bars->mma);
    }
    // the next item's K codes: their loads run under PV and the epilogue
    if (li + 1 < cnt) load_codes(page_of(li + 1), 0, tid, kc);
    ok = poll_wait(&bars->mma, 1, &bars->abort, p.wait_ns);
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();

    // 6. the partial: O / l in V's code units (the combine applies v_scale)
    if (warp_valid) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t ra[32], rb[32];
        tmem_ld32(tmem + lane_off + half * 64, ra);
        tmem_ld32(tmem + lane_off + half * 64 + 32, rb);
        tmem_wait_ld();
        if (valid)
          store_partial_half(ra, rb, inv, p.part_o + (int64_t)prow * kD + half * 64,
                             p.part_big + (int64_t)prow * (2 * kD) + half * 128,
                             p.e4m3_over4, pol_keep);
      }
      if (valid) {
        const float lse = l > 0.f ? (m2 + __log2f(l)) * 0.69314718055994530942f : -INFINITY;
        st_global_f32_hint(p.part_lse + prow, lse, pol_keep);
      }
    }
    tc_fence_before();
  }

  if (failed && tid == 0) {
    bars->abort = 1;
    atomicOr(p.status, (unsigned)MSA_STATUS_TIMEOUT);
  }
  cp_async_wait<0>();
  if (tid == 0) {
    // every MMA must complete before the CTA exits and frees its tensor
    // memory
    mma_commit(&bars->mma_done);
    bounded_wait(&bars->mma_done, 0, nullptr, kWaitLimitNs);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemColsB);
  }
}

}  // namespace

cudaError_t launch_attention_bf16q(const AttnArgs& a, cudaStream_t stream) {
  const msa_plan_t& pl = *a.plan;
  if (pl.max_work == 0) return cudaSuccess;
  ParamsB p;
  p.q16 = reinterpret_cast<const uint16_t*>(a.q);
  p.kv = a.kv;
  p.records = reinterpret_cast<const int4*>(pl.records);
  p.rec_stride = (int)(pl.record_bytes / 16);
  p.counters = pl.counters;
  p.part_o = a.part_o;
  p.part_big = a.part_big;
  p.part_vscale = a.part_vscale;
  p.part_lse = a.part_lse;
  p.e4m3_over4 = partial_over4(a.v_scale);
  p.status = pl.status;
  p.Hq = (int)pl.Hq;
  p.G = (int)(pl.Hq / pl.Hkv);
  p.score_log2 = a.score_log2;
  p.v_scale = a.v_scale;
  p.wait_ns = (uint32_t)std::min<uint64_t>(pipeline_wait_limit_ns(), kWaitLimitNs);

  // the dynamic shared-memory limit is a per-device function attribute
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> attr_set[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(attention_bf16q_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemB);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_set[dev].store(true, std::memory_order_release);
  }
  const int64_t grid = std::min<int64_t>(kCtasPerSm * (int64_t)num_sms(), pl.max_work);
  return launch_pdl(attention_bf16q_kernel, dim3((unsigned)grid), dim3(kThreadsB),
                    (size_t)kSmemB, stream, p);
}

}  // namespace msa
