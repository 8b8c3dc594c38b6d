// Block-sparse attention over the planned (KV head, page, token chunk) work
// items, for sm_103a: TMA page loads gathered through block_table, E4M3
// tensor-core MMAs (tcgen05, kind::f8f6f4) accumulating S = Q K^T and
// O = P V in tensor memory, softmax in registers with the probabilities
// rounded to E4M3, and one normalised partial (O, lse) per (token, query
// head, top-k slot).
//
// What it computes follows vLLM PR 60684 (Details / "Kernel capability":
// E4M3 query over E4M3 K/V with E4M3 QK and PV MMAs; Details / "Numerics":
// softmax probabilities rounded to E4M3; Details / "Scales": q scale folded
// into the softmax scale) and the vLLM docs for sparse_attention_msa
// (MiniMaxM3SparseMSAImpl.forward: sparse_atten_func over the k2q CSR,
// causal=True, page_table=block_table).  The kernel design is this
// library's own.
//
// One CTA per SM, persistent; work items are dealt round-robin (CTA b takes
// items b, b + grid, ...), because the plan emits the items of one heavily
// selected KV row next to each other.  Every work item has a record
// written by the plan: {KV row of the page in the pool, token count n,
// first key position, first query head} and, per token, {token id, query
// position, top-k slot}.  Warp roles (16 warps):
//   warp 0      producer: headers and token ids staged 8 items ahead in
//               shared memory by cp.async; bulk copy of the item's record;
//               TMA loads of the K and V halves of the page (2 x 16 KB,
//               128-byte swizzle) and, when G is a multiple of 8, of the Q
//               rows: one box of G rows per token, one lane per token
//   warp 1      tcgen05 issuer (one thread) and TMEM owner (512 columns)
//   warps 2-3   Q gather when G is not a multiple of 8: cp.async of 16-byte
//               chunks into the 128-byte-swizzled K-major tile
//   warps 4-7   softmax group 0 (even items)
//   warps 8-11  softmax group 1 (odd items)
//   warps 12-15 epilogue: O from TMEM, normalised, rounded to E4M3 in V's
//               code units (the combine applies v_scale), written as whole
//               32-byte sectors
// Shared memory: a 4-slot ring of {K, V} 16 KB tiles with the item's record
// (released when PV completes), a 3-slot ring of Q tiles (released when QK
// completes), 2 P tiles, and a 4-slot ring of per-row results handed from
// softmax to epilogue.
// TMEM: per group an S tile (128 columns) and an O tile (128 columns).
// The MMA thread issues QK(n) and PV(n) in order, each as soon as its inputs
// are ready.  QK(n) reuses the S tile of item n-2 as soon as the softmax
// holds S(n-2) in registers, so scores for the next items are computed
// while earlier softmaxes run.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kKvStages = 4;
constexpr int kQStages = 3;
constexpr int kTile = 128 * 128;  // one 128 x 128 E4M3 tile, bytes
constexpr int kThreads = 512;
constexpr int kSoftmaxThreads = 128;
constexpr int kTmemCols = 512;
constexpr int kRegsControl = 48;
constexpr int kRegsSoftmax = 176;
constexpr int kRegsEpilogue = 104;
static_assert(4 * 32 * kRegsControl + 8 * 32 * kRegsSoftmax +
                  4 * 32 * kRegsEpilogue <= 65536,
              "register split must equal the launch allocation");
constexpr int kRecMax = 16 * (1 + kTileM);  // header + up to 128 tokens

// offsets from the 1024-byte aligned base
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKvStages * kTile;
constexpr int kOffQ = kOffV + kKvStages * kTile;
constexpr int kOffP = kOffQ + kQStages * kTile;
constexpr int kOffRec = kOffP + 2 * kTile;
constexpr int kMetaSlots = 4;
// per row: partial row index (int64, -1 = none), lse, 1/l * v_scale
struct RowMeta {
  int64_t prow;
  float lse;
  float inv;
};
constexpr int kOffMeta = kOffRec + kKvStages * kRecMax;
// producer staging of prefetched record headers and token ids: two halves
// of kBatch items each
constexpr int kBatch = 8;
constexpr int kOffStage = kOffMeta + kMetaSlots * kTileM * (int)sizeof(RowMeta);
constexpr int kStageHdr = 2 * kBatch * 16;                   // int4 per item
constexpr int kStageTok = 2 * kBatch * 16 * 4;               // 16 ids per item
constexpr int kOffBar = kOffStage + kStageHdr + kStageTok;

struct Barriers {
  uint64_t rec_full[kKvStages];
  uint64_t kv_full[kKvStages];
  uint64_t kv_empty[kKvStages];
  uint64_t q_full[kQStages];
  uint64_t q_empty[kQStages];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t o_free[2];
  uint64_t meta_full[kMetaSlots];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

constexpr int kSmemBytes = kOffBar + (int)sizeof(Barriers) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory above the 227 KB limit");

struct Params {
  const uint8_t* q;
  const int4* records;
  int rec_stride;  // int4 per record
  const int32_t* counters;
  uint8_t* part_o;      // E4M3 partial rows, V's code units
  float* part_vscale;   // the combine's copy of v_scale
  float* part_lse;
  uint32_t* status;
  int Hq, G;
  int q_tma;       // 1: Q rows by TMA (G % 8 == 0), 0: by cp.async
  int rotate;      // 1: an item's rows rotate by (item % 4) * 32 (G divides 32)
  float inv_G;     // 1 / G, for div_G
  float score_log2;
  float v_scale;
};

__device__ __forceinline__ void set_timeout(Barriers* bars, uint32_t* status) {
  bars->abort = 1;
  atomicOr(status, (unsigned)MSA_STATUS_TIMEOUT);
}

// Rows of item li are placed rot(li) lanes further down the tile (mod 128)
// so that small items -- a few tokens x G heads, fewer than 32 rows -- land
// on a different TMEM lane quadrant, and so a different SM sub-partition,
// from one item to the next.  Only for G dividing 32: then a token's G rows
// start at a multiple of G and never straddle the end of the tile (a TMA
// box does not wrap around).
__device__ __forceinline__ int row_rotation(int li, int rotate) {
  return rotate ? (li & 3) * 32 : 0;
}

// lrow / G for 0 <= lrow < 128 and 1 <= G <= 128 by one multiply: the exact
// quotient (lrow + 0.5) / G lies at least 0.5 / G from an integer, far more
// than the float rounding error, so truncation gives the integer quotient.
__device__ __forceinline__ int div_G(int lrow, float inv_G) {
  return __float2int_rz(((float)lrow + 0.5f) * inv_G);
}

// p = 2^(x * c + off) for 32 score columns, packed to E4M3 in pairs and
// stored as two 16-byte chunks of the 128-byte-swizzled P row; returns the
// sum of the (unrounded) probabilities.  kMask: columns past kv_lim are 0.
// Four floats rounded to E4M3 (nearest even, saturating) in one word, the
// first in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

template <bool kMask>
__device__ __forceinline__ float exp_pack32(const uint32_t (&r)[32], int col0,
                                            int kv_lim, float c, float off,
                                            uint8_t* prow, int row) {
  uint32_t packed[8];
  float l = 0.f;
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    float pv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float x = __uint_as_float(r[e + u]);
      pv[u] = ex2_approx(fmaf(x, c, off));
      if (kMask && col0 + e + u > kv_lim) pv[u] = 0.f;
      l += pv[u];
    }
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(pv[0], pv[1]),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(pv[2], pv[3]),
                                                 __NV_SATFINITE, __NV_E4M3);
    packed[e / 4] = lo | (hi << 16);
  }
  const int c0 = col0 / 16, c1 = c0 + 1;
  *reinterpret_cast<uint4*>(prow + ((c0 ^ (row & 7)) << 4)) =
      make_uint4(packed[0], packed[1], packed[2], packed[3]);
  *reinterpret_cast<uint4*>(prow + ((c1 ^ (row & 7)) << 4)) =
      make_uint4(packed[4], packed[5], packed[6], packed[7]);
  return l;
}

template <bool kMask>
__device__ __forceinline__ float max32(const uint32_t (&r)[32], int col0,
                                       int kv_lim, float m) {
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float x = __uint_as_float(r[e]);
    if (!kMask || col0 + e <= kv_lim) m = fmaxf(m, x);
  }
  return m;
}

__global__ void __launch_bounds__(kThreads, 1)
attention_kernel(const __grid_constant__ CUtensorMap kv_map,
                 const __grid_constant__ CUtensorMap q_map, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kOffBar);
  const volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // the plan's counters and records are written by the kernels before this
  // one in the stream
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.part_vscale = p.v_scale;
  const int num_work = p.counters[1];
  // work items are dealt round-robin: CTA b takes items b, b + grid, ...
  // Items of one heavily selected KV row are adjacent in the work list, so
  // contiguous ranges would give a few CTAs all of the full 128-row items.
  const int cnt = blockIdx.x < (unsigned)num_work
                      ? (num_work - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                      : 0;
  const int64_t rec_step = (int64_t)gridDim.x * p.rec_stride;  // int4s between own items

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(&bars->rec_full[s], 1);
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&bars->q_full[s], p.q_tma ? 1 : 32);
      mbar_init(&bars->q_empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&bars->s_full[w], 1);
      mbar_init(&bars->s_free[w], kSoftmaxThreads);
      mbar_init(&bars->p_full[w], kSoftmaxThreads);
      mbar_init(&bars->o_full[w], 1);
      mbar_init(&bars->o_free[w], kSoftmaxThreads);
    }
    for (int m = 0; m < kMetaSlots; ++m)
      mbar_init(&bars->meta_full[m], kSoftmaxThreads);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // Launched with 128 registers per thread (512 threads); each role's
  // warpgroup then resizes: softmax 176, epilogue 104, control warps 48
  // (4*32*48 + 8*32*176 + 4*32*104 = 64512 <= 65536).

  if (warp < 4) {
  setmaxnreg_dec<kRegsControl>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // whole warp: lane 0 waits for free slots and issues the record / K / V
    // copies; in TMA-Q mode lane i issues the Q box of the item's token i
    // (C = 128 / G <= 16 tokens).
    const int4* grec = p.records + (int64_t)blockIdx.x * p.rec_stride;
    const int C = kTileM / p.G;
    // Headers and token ids are staged kBatch items ahead in shared memory
    // by cp.async: the copies of batch b+1 are issued when batch b starts and
    // waited for when it ends, so the producer never stalls on a global
    // load.  Lane j < kBatch copies the header of item j; lane l copies the
    // token ids at flat entries l, l+32, l+64, l+96 of the kBatch x 16 ids.
    int4* shdr = reinterpret_cast<int4*>(smem + kOffStage);
    int* stok = reinterpret_cast<int*>(smem + kOffStage + kStageHdr);
    auto load_batch = [&](int base, int half) {
      if (lane < kBatch && base + lane < cnt)
        cp_async_16(smem_u32(shdr + half * kBatch + lane),
                    grec + (base + lane) * rec_step);
      if (p.q_tma) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = lane + 32 * u, j = e >> 4, i = e & 15;
          if (i < C && base + j < cnt)
            cp_async_4(smem_u32(stok + half * kBatch * 16 + e),
                       grec + (base + j) * rec_step + 1 + i);
        }
      }
      cp_async_commit();
    };
    auto wait_batch = [&]() {
      cp_async_wait<0>();
      __syncwarp();
    };
    load_batch(0, 0);
    wait_batch();
    int issued = 0;
    bool ok_all = true;
    for (int base = 0; ok_all && base < cnt; base += kBatch) {
      const int half = (base / kBatch) & 1;
      if (base + kBatch < cnt) load_batch(base + kBatch, half ^ 1);
      for (int j = 0; j < kBatch && base + j < cnt; ++j) {
        const int li = base + j;
        const int ks = li % kKvStages, qs = li % kQStages;
        const int4 hdr = shdr[half * kBatch + j];
        const int tok = (lane < 16) ? stok[(half * kBatch + j) * 16 + lane] : 0;
        int ok = 1;
        if (lane == 0) {
          if (li >= kKvStages)
            ok = bounded_wait(&bars->kv_empty[ks], ((li / kKvStages) - 1) & 1,
                              abort, kWaitLimitNs);
          if (ok && li >= kQStages)
            ok = bounded_wait(&bars->q_empty[qs], ((li / kQStages) - 1) & 1,
                              abort, kWaitLimitNs);
          if (!ok && !*abort) set_timeout(bars, p.status);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          ok_all = false;
          break;
        }
        if (lane == 0) {
          const uint32_t rec_bytes = 16u * (1u + (uint32_t)hdr.y);
          mbar_arrive_expect_tx(&bars->rec_full[ks], rec_bytes);
          bulk_load(smem + kOffRec + ks * kRecMax,
                    grec + li * rec_step, rec_bytes,
                    &bars->rec_full[ks]);
          mbar_arrive_expect_tx(&bars->kv_full[ks], 2 * kTile);
          tma_load_2d(smem + kOffK + ks * kTile, &kv_map, &bars->kv_full[ks], 0, hdr.x);
          tma_load_2d(smem + kOffV + ks * kTile, &kv_map, &bars->kv_full[ks], kD, hdr.x);
          if (p.q_tma)
            mbar_arrive_expect_tx(&bars->q_full[qs], (uint32_t)(hdr.y * p.G * 128));
        }
        if (p.q_tma) {
          __syncwarp();
          if (lane < hdr.y)
            tma_load_2d(smem + kOffQ + qs * kTile +
                            ((lane * p.G + row_rotation(li, p.rotate)) & (kTileM - 1)) * 128,
                        &q_map, &bars->q_full[qs], 0, tok * p.Hq + hdr.w);
        }
        issued = li + 1;
      }
      // the other half is complete once this lane's copies have landed
      // and every lane is past this point
      if (base + kBatch < cnt) wait_batch();
    }
    cp_async_wait<0>();
    // every copy this warp started must land before the CTA exits
    if (lane == 0) {
      for (int li = issued > kKvStages ? issued - kKvStages : 0; li < issued; ++li) {
        bounded_wait(&bars->rec_full[li % kKvStages], (li / kKvStages) & 1,
                     nullptr, kWaitLimitNs);
        bounded_wait(&bars->kv_full[li % kKvStages], (li / kKvStages) & 1,
                     nullptr, kWaitLimitNs);
      }
      if (p.q_tma)
        for (int li = issued > kQStages ? issued - kQStages : 0; li < issued; ++li)
          bounded_wait(&bars->q_full[li % kQStages], (li / kQStages) & 1,
                       nullptr, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_e4m3_f32(128, 128, false);
      constexpr uint32_t idesc_pv = idesc_e4m3_f32(128, 128, true);
      bool ok = true;
      auto issue_qk = [&](int li) {
        const int ks = li % kKvStages, qs = li % kQStages, w = li & 1;
        tc_fence_after();
        const uint64_t a = smem_desc_sw128(smem_u32(smem + kOffQ + qs * kTile), 16, 1024);
        const uint64_t b = smem_desc_sw128(smem_u32(smem + kOffK + ks * kTile), 16, 1024);
        const uint32_t d = tmem + (uint32_t)(w * 256);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // K = 128 bytes = 4 x 32
          mma_f8f6f4(d, a + (uint64_t)(kk * 2), b + (uint64_t)(kk * 2), idesc_qk,
                     kk > 0);
        mma_commit(&bars->s_full[w]);
        mma_commit(&bars->q_empty[qs]);
      };
      auto issue_pv = [&](int li) {
        const int ks = li % kKvStages, w = li & 1;
        tc_fence_after();
        const uint64_t a = smem_desc_sw128(smem_u32(smem + kOffP + w * kTile), 16, 1024);
        const uint64_t b = smem_desc_sw128(smem_u32(smem + kOffV + ks * kTile), 1024, 1024);
        const uint32_t d = tmem + (uint32_t)(w * 256 + 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 128 keys = 4 x 32; V rows advance 4 KB
          mma_f8f6f4(d, a + (uint64_t)(kk * 2), b + (uint64_t)(kk * 256),
                     idesc_pv, kk > 0);
        mma_commit(&bars->o_full[w]);
        mma_commit(&bars->kv_empty[ks]);
      };
      // in-order issue of QK(qk) and PV(pv), each as soon as it is ready;
      // QK(n) reuses the S tile of item n-2, free once the softmax has
      // loaded S(n-2) into registers
      int qk = 0, pv = 0;
      uint64_t idle_since = global_timer_ns();
      while (pv < cnt) {
        bool progressed = false;
        if (qk < cnt) {
          const int k = qk >> 1;
          if ((k == 0 || mbar_test(&bars->s_free[qk & 1], (k - 1) & 1)) &&
              mbar_test(&bars->kv_full[qk % kKvStages], (qk / kKvStages) & 1) &&
              mbar_test(&bars->q_full[qk % kQStages], (qk / kQStages) & 1)) {
            issue_qk(qk);
            ++qk;
            progressed = true;
          }
        }
        if (pv < qk) {
          const int w = pv & 1, k = pv >> 1;
          if (mbar_test(&bars->p_full[w], k & 1) &&
              (k == 0 || mbar_test(&bars->o_free[w], (k - 1) & 1))) {
            issue_pv(pv);
            ++pv;
            progressed = true;
          }
        }
        if (progressed) {
          idle_since = global_timer_ns();
        } else if (*abort || global_timer_ns() - idle_since > kWaitLimitNs) {
          ok = false;
          break;
        }
      }
      if (!ok && !*abort) set_timeout(bars, p.status);
      mma_commit(&bars->mma_done);
      bounded_wait(&bars->mma_done, 0, nullptr, kWaitLimitNs);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ Q gather
    // (cp.async mode only) two warps take alternate items; 16-byte chunks
    // into the swizzled layout, then a proxy fence so the tensor cores see
    // the rows.
    if (!p.q_tma) {
      bool ok = true;
      for (int li = warp - 2; li < cnt; li += 2) {
        const int ks = li % kKvStages, qs = li % kQStages;
        if (!bounded_wait(&bars->rec_full[ks], (li / kKvStages) & 1, abort,
                          kWaitLimitNs) ||
            (li >= kQStages &&
             !bounded_wait(&bars->q_empty[qs], ((li / kQStages) - 1) & 1, abort,
                           kWaitLimitNs))) {
          ok = false;
          break;
        }
        const int4* rec = reinterpret_cast<const int4*>(smem + kOffRec + ks * kRecMax);
        const int4 hdr = rec[0];
        const int rows = hdr.y * p.G;
        const int rot = row_rotation(li, p.rotate);
        const uint32_t dst0 = smem_u32(smem + kOffQ + qs * kTile);
        for (int e = lane; e < rows * 8; e += 32) {
          const int lrow = e >> 3, ch = e & 7;
          const int i = div_G(lrow, p.inv_G), g = lrow - i * p.G;
          const int row = (lrow + rot) & (kTileM - 1);
          const int t = rec[1 + i].x;
          const uint8_t* src =
              p.q + ((int64_t)t * p.Hq + hdr.w + g) * kD + ch * 16;
          cp_async_16(dst0 + row * 128 + ((ch ^ (row & 7)) << 4), src);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        mbar_arrive(&bars->q_full[qs]);
      }
      cp_async_wait<0>();
      if (!ok && lane == 0 && !*abort) set_timeout(bars, p.status);
    }
  }
  } else if (warp < 12) {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int w = (warp - 4) >> 2;       // group
    const int quad = warp & 3;           // TMEM lane quadrant
    const int row = quad * 32 + lane;    // tile row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + (uint32_t)(w * 256);
    uint8_t* prow_s = smem + kOffP + w * kTile + row * 128;
    RowMeta* meta = reinterpret_cast<RowMeta*>(smem + kOffMeta);
    for (int k = 0;; ++k) {
      const int li = 2 * k + w;
      if (li >= cnt) break;
      const int ks = li % kKvStages;
      if (!bounded_wait(&bars->rec_full[ks], (li / kKvStages) & 1, abort,
                        kWaitLimitNs)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      const int4* rec = reinterpret_cast<const int4*>(smem + kOffRec + ks * kRecMax);
      const int4 hdr = rec[0];
      // logical row (token i, head g) held by this lane for this item
      const int lrow = (row - row_rotation(li, p.rotate)) & (kTileM - 1);
      const int i = div_G(lrow, p.inv_G), g = lrow - i * p.G;
      const bool valid = i < hdr.y;
      const bool warp_valid = __any_sync(0xffffffffu, valid);
      int64_t prow = -1;
      int kv_lim = 127;
      if (valid) {
        const int4 tok = rec[1 + i];
        prow = ((int64_t)tok.x * p.Hq + hdr.w + g) * kTopK + tok.z;
        kv_lim = min(tok.y - hdr.z, 127);
      }
      const bool need_mask = __any_sync(0xffffffffu, valid && kv_lim < 127);
      if (!bounded_wait(&bars->s_full[w], k & 1, abort, kWaitLimitNs)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      if (warp_valid) {
        __syncwarp();
        tmem_ld32(s_tmem + 0, r0);
        tmem_ld32(s_tmem + 32, r1);
        tmem_ld32(s_tmem + 64, r2);
        tmem_ld32(s_tmem + 96, r3);
        tmem_wait_ld();
      }
      // S is in registers: QK of this group's next item may overwrite it
      tc_fence_before();
      mbar_arrive(&bars->s_free[w]);
      // the P tile is free once PV of this group's previous item is done
      if (k > 0 &&
          !bounded_wait(&bars->o_full[w], (k - 1) & 1, abort, kWaitLimitNs)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      float m2 = -INFINITY, l = 0.f;
      if (warp_valid) {
        float m = -INFINITY;
        if (need_mask) {
          m = max32<true>(r0, 0, kv_lim, m);
          m = max32<true>(r1, 32, kv_lim, m);
          m = max32<true>(r2, 64, kv_lim, m);
          m = max32<true>(r3, 96, kv_lim, m);
        } else {
          m = max32<false>(r0, 0, kv_lim, m);
          m = max32<false>(r1, 32, kv_lim, m);
          m = max32<false>(r2, 64, kv_lim, m);
          m = max32<false>(r3, 96, kv_lim, m);
        }
        m2 = m * p.score_log2;
        // p = 2^(x * c - m2 + 8): probabilities scaled by 256 so that small
        // ones stay out of E4M3's subnormal range; l and O carry the same
        // factor, which cancels.
        const float off = (m2 == -INFINITY) ? 0.f : 8.f - m2;
        const float c = p.score_log2;
        if (need_mask) {
          l += exp_pack32<true>(r0, 0, kv_lim, c, off, prow_s, row);
          l += exp_pack32<true>(r1, 32, kv_lim, c, off, prow_s, row);
          l += exp_pack32<true>(r2, 64, kv_lim, c, off, prow_s, row);
          l += exp_pack32<true>(r3, 96, kv_lim, c, off, prow_s, row);
        } else {
          l += exp_pack32<false>(r0, 0, kv_lim, c, off, prow_s, row);
          l += exp_pack32<false>(r1, 32, kv_lim, c, off, prow_s, row);
          l += exp_pack32<false>(r2, 64, kv_lim, c, off, prow_s, row);
          l += exp_pack32<false>(r3, 96, kv_lim, c, off, prow_s, row);
        }
      }
      RowMeta mt;
      mt.prow = prow;
      mt.inv = l > 0.f ? 1.f / l : 0.f;  // O in V's code units; the combine scales
      mt.lse = l > 0.f ? (m2 + __log2f(l) - 8.f) * 0.69314718055994530942f
                       : -INFINITY;
      meta[(li % kMetaSlots) * kTileM + row] = mt;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full[w]);
      mbar_arrive(&bars->meta_full[li % kMetaSlots]);
    }
  } else {
    setmaxnreg_dec<kRegsEpilogue>();
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const RowMeta* meta = reinterpret_cast<const RowMeta*>(smem + kOffMeta);
    for (int li = 0; li < cnt; ++li) {
      const int w = li & 1, k = li >> 1;
      if (!bounded_wait(&bars->meta_full[li % kMetaSlots],
                        (li / kMetaSlots) & 1, abort, kWaitLimitNs)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      const RowMeta mt = meta[(li % kMetaSlots) * kTileM + row];
      const bool valid = mt.prow >= 0;
      const bool warp_valid = __any_sync(0xffffffffu, valid);
      if (!bounded_wait(&bars->o_full[w], k & 1, abort, kWaitLimitNs)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      tc_fence_after();
      if (warp_valid) {
        const uint32_t o_tmem = tmem + lane_off + (uint32_t)(w * 256 + 128);
        uint8_t* dst = p.part_o + mt.prow * (int64_t)kD;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t ra[32], rb[32];
          __syncwarp();
          tmem_ld32(o_tmem + half * 64, ra);
          tmem_ld32(o_tmem + half * 64 + 32, rb);
          tmem_wait_ld();
          if (valid) {
            // the normalised row in V's code units is a convex combination
            // of E4M3 V codes, so it stays within E4M3's range; word k holds
            // columns 4k .. 4k+3 of this half
            uint32_t o[16];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              o[k] = pack_e4m3x4(__uint_as_float(ra[4 * k]) * mt.inv,
                                 __uint_as_float(ra[4 * k + 1]) * mt.inv,
                                 __uint_as_float(ra[4 * k + 2]) * mt.inv,
                                 __uint_as_float(ra[4 * k + 3]) * mt.inv);
              o[8 + k] = pack_e4m3x4(__uint_as_float(rb[4 * k]) * mt.inv,
                                     __uint_as_float(rb[4 * k + 1]) * mt.inv,
                                     __uint_as_float(rb[4 * k + 2]) * mt.inv,
                                     __uint_as_float(rb[4 * k + 3]) * mt.inv);
            }
            // whole 32-byte sectors: the row's half is 64 bytes at a
            // 64-byte aligned offset of a 128-byte row
            uint8_t* d = dst + half * 64;
            st_global_v8(d, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
            st_global_v8(d + 32, o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15]);
          }
        }
        if (valid) p.part_lse[mt.prow] = mt.lse;
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free[w]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                   void*, const cuuint64_t*, const cuuint64_t*,
                                   const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// A 2-D byte tensor of `rows` rows of `row_bytes`, read in boxes of
// box_rows x 128 bytes with the 128-byte swizzle the MMA descriptors expect.
bool encode_rows(EncodeTiledFn enc, CUtensorMap* map, const void* base,
                 uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  const msa_plan_t& pl = *a.plan;
  if (pl.max_work == 0) return cudaSuccess;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int G = (int)(pl.Hq / pl.Hkv);
  // page pool: rows = (page, KV head, token), 256 bytes each (K then V)
  CUtensorMap kv_map, q_map;
  if (!encode_rows(enc, &kv_map, a.kv, 2 * kD,
                   (uint64_t)a.num_pages * pl.Hkv * kPage, 128))
    return cudaErrorInvalidValue;
  // queries: rows = (token, query head), 128 bytes each; one box = the G
  // heads of one KV head of one token
  const bool q_tma = (G % 8) == 0;
  if (q_tma) {
    if (!encode_rows(enc, &q_map, a.q, kD, (uint64_t)pl.T * pl.Hq, (uint32_t)G))
      return cudaErrorInvalidValue;
  } else {
    q_map = kv_map;  // unused
  }

  Params p;
  p.q = a.q;
  p.records = reinterpret_cast<const int4*>(pl.records);
  p.rec_stride = (int)(pl.record_bytes / 16);
  p.counters = pl.counters;
  p.part_o = a.part_o;
  p.part_vscale = a.part_vscale;
  p.part_lse = a.part_lse;
  p.status = pl.status;
  p.Hq = (int)pl.Hq;
  p.G = G;
  p.rotate = (G <= 32 && 32 % G == 0) ? 1 : 0;
  p.inv_G = 1.0f / (float)G;
  p.q_tma = q_tma ? 1 : 0;
  p.score_log2 = a.score_log2;
  p.v_scale = a.v_scale;

  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t grid = std::min<int64_t>(num_sms(), pl.max_work);
  return launch_pdl(attention_kernel, dim3((unsigned)grid), dim3(kThreads), kSmemBytes,
                    stream, kv_map, q_map, p);
}

}  // namespace msa
