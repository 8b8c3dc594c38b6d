// Block-sparse attention over the planned (KV head, page, token chunk) work
// items, for sm_103a: TMA page loads gathered through block_table, E4M3
// tensor-core MMAs (tcgen05, kind::f8f6f4) accumulating S = Q K^T and
// O = P V in tensor memory, softmax in registers with the probabilities
// rounded to E4M3, and one normalised partial (O, lse) per (token, query
// head, top-k slot).
//
// What it computes follows vLLM PR 60684 (Details / "Kernel capability":
// E4M3 query over E4M3 K/V with E4M3 QK and PV MMAs, and over NVFP4 K/V
// with each code times its block scale dequantised to E4M3; Details /
// "Numerics": softmax probabilities rounded to E4M3; Details / "Scales":
// q scale folded into the softmax scale) and the vLLM docs for
// sparse_attention_msa (MiniMaxM3SparseMSAImpl.forward: sparse_atten_func
// over the k2q CSR, causal=True, page_table=block_table).  The kernel design
// is this library's own.
//
// One CTA per SM, persistent; work items are dealt round-robin (CTA b takes
// items b, b + grid, ...), because the plan emits the items of one heavily
// selected KV row next to each other.  Every work item has a record
// written by the plan: {KV row of the page in the pool, token count n,
// first key position, first query head} and, per token, {token id, query
// position, top-k slot}.  Warp roles (16 warps):
//   warp 0      producer: headers and token ids staged 8 items ahead in
//               shared memory by cp.async; bulk copy of the item's record;
//               E4M3 pool: TMA loads of the K and V halves of the page
//               (2 x 16 KB, 128-byte swizzle); NVFP4 pool: bulk copies of
//               the page-head's K and V slots (2 x 9 KB); and, when G is a
//               multiple of 8, TMA loads of the Q rows: one box of G rows
//               per token, one lane per token
//   warp 1      tcgen05 issuer (one thread) and TMEM owner (512 columns)
//   warps 2-3   Q gather when G is not a multiple of 8: cp.async of 16-byte
//               chunks into the 128-byte-swizzled K-major tile; NVFP4: also
//               the dequantisation of each item's V slot
//   warps 4-7   softmax group 0 (even items)
//   warps 8-11  softmax group 1 (odd items); NVFP4: each group also
//               dequantises the K slot of its next item after writing P
//   warps 12-15 epilogue: O from TMEM, normalised, rounded to E4M3 in V's
//               code units (the combine applies v_scale), written as whole
//               32-byte sectors
// Shared memory (E4M3 pool): a 3-slot ring of K tiles (16 KB, released when
// QK completes), a ring of V tiles with the item's record (released when PV
// completes) and a ring of Q/P tiles, 5 deep on sparse plans and 3 on dense
// ones (Ring below) -- the item's Q rows,
// which its softmax overwrites with P once QK has completed (released when
// PV completes) -- and a ring of per-row results handed from softmax to
// epilogue.  K leaves shared memory as soon as the scores are computed, so
// more V and Q/P tiles fit, and those are the ones held through the
// softmax.  The NVFP4 layout is described at Ring below.
// TMEM: per group an S tile (128 columns) and an O tile (128 columns).
// The MMA thread issues QK(n) and PV(n) in order, each as soon as its inputs
// are ready.  QK(n) reuses the S tile of item n-2 as soon as the softmax
// holds S(n-2) in registers, so scores for the next items are computed
// while earlier softmaxes run.  Because every item writes P into its own
// slot, the softmax of item n never waits for PV of item n-2: the items of
// one group, whose rows sit in different TMEM lane quadrants, are worked on
// by different warps at the same time.
#include <cuda.h>
#include <atomic>
#include <cmath>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "nvfp4.cuh"
#include "partial.cuh"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kTile = 128 * 128;  // one 128 x 128 E4M3 tile, bytes
constexpr int kThreads = 512;
constexpr int kSoftmaxThreads = 128;
constexpr int kTmemCols = 512;
constexpr int kRegsControl = 64;
constexpr int kRegsSoftmax = 176;
constexpr int kRegsEpilogue = 96;
static_assert(4 * 32 * kRegsControl + 8 * 32 * kRegsSoftmax +
                  4 * 32 * kRegsEpilogue <= 65536,
              "register split must equal the launch allocation");
constexpr int kRecMax = 16 * (1 + kTileM);  // header + up to 128 tokens
constexpr int kMetaSlots = 3;
// per row: partial row index (-1 = none; below 2^31, the host checks
// T * Hq * 16 against it), lse, 1/l
struct RowMeta {
  int32_t prow;
  float lse;
  float inv;
};
// producer staging of prefetched record headers and token ids: two halves
// of kBatch items each
constexpr int kBatch = 8;
constexpr int kStageHdr = 2 * kBatch * 16;                   // int4 per item
constexpr int kStageTok = 2 * kBatch * 16 * 4;               // 16 ids per item
// L2 policy hints: K/V pages are read once (evict first); Q rows are read by
// every item of their tokens and the partials by the combine (evict last).
// (Prefetching the next items' pages into L2 with bulk prefetches was
// measured slower: the prefetches queue in the same TMA unit as the loads.)

constexpr int kMaxRing = 6;
struct Barriers {
  uint64_t rec_full[kMaxRing];
  uint64_t kraw_full[kMaxRing];  // NVFP4: K slot of the page-head landed
  uint64_t kraw_empty[kMaxRing]; // NVFP4: K slot converted
  uint64_t vraw_full[kMaxRing];  // NVFP4: V slot landed
  uint64_t vraw_empty[kMaxRing]; // NVFP4: V slot converted
  uint64_t k_full[kMaxRing];     // K tile ready (landed, or converted)
  uint64_t v_full[kMaxRing];     // V tile ready (landed, or converted)
  uint64_t v_empty[kMaxRing];    // PV done, the V tile is free
  uint64_t k_empty[kMaxRing];    // QK done, the K tile is free
  uint64_t q_full[kMaxRing];
  uint64_t q_empty[kMaxRing];    // PV done: the Q/P slot is free
  uint64_t p_full[kMaxRing];     // P of the slot's item written
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t o_full[2];
  uint64_t o_free[2];
  uint64_t meta_full[kMetaSlots];
  uint64_t meta_free[kMetaSlots];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

// Shared-memory rings and offsets from the 1024-byte aligned base.
//   E4M3 pool: 3 K tiles and 5 V tiles filled by TMA, then 5 Q/P slots;
//   the record ring (one record per V slot) follows the tile rings.
//   NVFP4 pool: the K and V slots of a page-head (9 KB each) land in rings
//   of 3 each; the softmax group of item j - 2 converts K slot j once it has
//   written P(j - 2), warps 2-3 convert V slot j once PV(j - 2) is done;
//   then 2 K and 2 V E4M3 tiles, 4 Q/P slots and the 2 KB code x scale
//   lookup table.  A record is read until its softmax starts, which
//   precedes the conversion of the K and V slots two items later, so a ring
//   of min(K slots, V slots) + 2 records never overwrites one in use.
// kDepth: the E4M3 pool's V and Q/P ring depth, 5 for sparse plans and 3
// for dense ones.  Measured on GB300 in whole steps (plan, attention and
// combine chained), with the warp roles in their earlier order in the code
// (control warps first): 5 is 3-4 us faster than 4 on long_prefill_1m and the
// 64-request decode; on long_prefill_150k and the ragged batch 4 is
// 14-15 us faster than 5 and 3 another 4-5 us faster than 4, while 2 is
// 40 us slower; the NVFP4 pool has rings of its own.
template <bool kFp4, int kDepth>
struct Ring {
  static constexpr int k = kFp4 ? 2 : 3;  // K tiles (free once QK is done)
  static constexpr int v = kFp4 ? 2 : kDepth;  // V tiles (free once PV is done)
  static constexpr int kraw = kFp4 ? 3 : 0;
  static constexpr int vraw = kFp4 ? 3 : 0;
  static constexpr int q = kFp4 ? 4 : kDepth;  // Q/P slots: P(n) overwrites Q(n)
  static constexpr int rec = kFp4 ? (kraw < vraw ? kraw : vraw) + 2 : v;
  static constexpr int off_k = 0;
  static constexpr int off_v = off_k + k * kTile;
  static constexpr int off_q = off_v + v * kTile;
  static constexpr int off_kraw = off_q + q * kTile;
  static constexpr int off_vraw = off_kraw + kraw * kFp4Slot;
  static constexpr int off_lut = off_vraw + vraw * kFp4Slot;
  static constexpr int off_rec = off_lut + (kFp4 ? kFp4LutBytes : 0);
  static constexpr int off_meta = off_rec + rec * kRecMax;
  static constexpr int off_stage =
      off_meta + kMetaSlots * kTileM * (int)sizeof(RowMeta);
  static constexpr int off_bar = off_stage + kStageHdr + kStageTok;
  static constexpr int bytes = off_bar + (int)sizeof(Barriers) + 1024;
  static_assert(rec <= kMaxRing && q <= kMaxRing && k <= kMaxRing && v <= kMaxRing &&
                    kraw <= kMaxRing && vraw <= kMaxRing,
                "ring deeper than the barrier arrays");
  static_assert(off_rec % 16 == 0 && off_kraw % 16 == 0 && off_vraw % 16 == 0 &&
                    kFp4Slot % 16 == 0 && off_meta % 4 == 0 && off_stage % 16 == 0,
                "bulk-copy destinations must be 16-byte aligned");
  static_assert(bytes <= 232448, "shared memory above the 227 KB limit");
};

struct Params {
  const uint8_t* q;
  const uint8_t* kv4;   // NVFP4 pool (page-heads of kFp4PageHead bytes)
  const int4* records;
  int rec_stride;  // int4 per record
  const int32_t* counters;
  uint8_t* part_o;      // E4M3 partial rows, V's code units, 128 bytes each
  uint8_t* part_big;    // bf16 overflow rows, 256 bytes each
  float* part_vscale;   // the combine's copy of v_scale
  float* part_lse;
  uint32_t e4m3_over4;  // (0x7F - largest E4M3 magnitude code a half keeps)
                        // in each byte
  uint32_t* status;
  int Hq, G;
  int q_tma;       // 1: Q rows by TMA (G % 8 == 0), 0: by cp.async
  int rotate;      // 1: an item's rows rotate by (item % 4) * 32 (G divides 32)
  float inv_G;     // 1 / G, for div_G
  float score_log2;
  float v_scale;
  // wall-time limit of the pipeline waits, in ns (the drains of copies and
  // MMAs in flight before a CTA exits always keep kWaitLimitNs)
  uint32_t wait_ns;
};

// bounded_wait taken by a whole warp: every lane waits, and the warp goes on
// only if every lane saw the phase complete, so that on a timeout the lanes
// of a warp never part ways before a warp-wide step (a shuffle, a vote, a
// tcgen05.ld or a __syncwarp)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          const volatile int* abort, uint32_t limit_ns) {
  return __all_sync(0xffffffffu, bounded_wait(bar, parity, abort, limit_ns));
}

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
// stored as two 16-byte chunks of the 128-byte-swizzled P row; adds the
// (unrounded) probabilities to four independent partial sums (column
// e % 4 to l[e % 4]), so the additions form four short chains instead of
// one long one.  Masked columns hold -inf and give 0.
__device__ __forceinline__ void exp_pack32(const uint32_t (&r)[32], int col0, float c,
                                           float off, uint8_t* prow, int row, float (&l)[4]) {
  uint32_t packed[8];
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    float pv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float x = __uint_as_float(r[e + u]);
      pv[u] = ex2_approx(fmaf(x, c, off));
      l[u] += pv[u];
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
}

// Row maximum over 32 score columns into four independent partial maxima
// (column e % 4 to m[e % 4]): four short dependency chains.
__device__ __forceinline__ void max32(const uint32_t (&r)[32], float (&m)[4]) {
#pragma unroll
  for (int e = 0; e < 32; ++e) m[e & 3] = fmaxf(m[e & 3], __uint_as_float(r[e]));
}

// The causal mask of an item on the token's own page: the score columns past
// kv_lim become -inf, so that the one unmasked code path serves every item
// (a second, masked copy of the max and exponential loops would not fit the
// instruction cache beside the other warp roles' loops).
__device__ __forceinline__ void mask32(uint32_t (&r)[32], int col0, int kv_lim) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (col0 + e > kv_lim) r[e] = 0xFF800000u;
}

// One 128-token slot (K or V) of an NVFP4 page-head, dequantised into a
// 128 x 128 E4M3 tile in the 128-byte-swizzled layout a TMA box would have
// written: 1024 blocks of 16 elements, thread c of kN threads taking blocks
// c, c + kN, ...  Code loads are 8 contiguous bytes per thread and the
// 16-byte stores of a warp cover 4 whole rows, so neither has bank
// conflicts.
// Blocks go in batches of four whose loads are all issued before any of
// their stores, so the shared-memory latencies of a batch overlap (the
// compiler cannot move a load above a store to the same array itself).
template <int kN>
__device__ __forceinline__ void convert_slot(const uint8_t* raw, uint8_t* tile,
                                             const uint8_t* lut, int c) {
  constexpr int kBatchBlocks = 4;
  static_assert((1024 / kN) % kBatchBlocks == 0, "whole batches per thread");
#pragma unroll 1
  for (int j = 0; j < 1024 / kN; j += kBatchBlocks) {
    uint2 codes[kBatchBlocks];
    uint32_t scale[kBatchBlocks];
#pragma unroll
    for (int u = 0; u < kBatchBlocks; ++u) {
      const int blk = (j + u) * kN + c;
      codes[u] = *reinterpret_cast<const uint2*>(raw + blk * 8);
      scale[u] = raw[kFp4Codes + blk];
    }
    uint4 out[kBatchBlocks];
#pragma unroll
    for (int u = 0; u < kBatchBlocks; ++u)
      out[u] = nvfp4_block_to_e4m3(codes[u], scale[u], lut);
#pragma unroll
    for (int u = 0; u < kBatchBlocks; ++u) {
      const int blk = (j + u) * kN + c, t = blk >> 3, b = blk & 7;
      *reinterpret_cast<uint4*>(tile + t * 128 + ((b ^ (t & 7)) << 4)) = out[u];
    }
  }
}

template <bool kFp4, int kDepth>
__global__ void __launch_bounds__(kThreads, 1)
attention_kernel(const __grid_constant__ CUtensorMap kv_map,
                 const __grid_constant__ CUtensorMap q_map, const Params p) {
  using L = Ring<kFp4, kDepth>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Barriers* bars = reinterpret_cast<Barriers*>(smem + L::off_bar);
  const volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // the plan's counters and records are written by the kernels before this
  // one in the stream
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.part_vscale = p.v_scale;
  // a plan whose construction timed out is incomplete: no work
  const int num_work = (*p.status & MSA_STATUS_TIMEOUT) ? 0 : p.counters[1];
  // work items are dealt round-robin: CTA b takes items b, b + grid, ...
  // Items of one heavily selected KV row are adjacent in the work list, so
  // contiguous ranges would give a few CTAs all of the full 128-row items.
  const int cnt = blockIdx.x < (unsigned)num_work
                      ? (num_work - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                      : 0;
  const int64_t rec_step = (int64_t)gridDim.x * p.rec_stride;  // int4s between own items

  if (threadIdx.x == 0) {
    // NVFP4: each converting warp arrives once (lane 0, after a
    // __syncwarp): the four warps of a softmax group on k_full and
    // kraw_empty; warps 2-3 on v_full, vraw_empty and, gathering Q, q_full
    for (int s = 0; s < L::rec; ++s) mbar_init(&bars->rec_full[s], 1);
    for (int s = 0; s < L::kraw; ++s) {
      mbar_init(&bars->kraw_full[s], 1);
      mbar_init(&bars->kraw_empty[s], 4);
    }
    for (int s = 0; s < L::vraw; ++s) {
      mbar_init(&bars->vraw_full[s], 1);
      mbar_init(&bars->vraw_empty[s], 2);
    }
    for (int s = 0; s < L::k; ++s) {
      mbar_init(&bars->k_full[s], kFp4 ? 4 : 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < L::v; ++s) {
      mbar_init(&bars->v_full[s], kFp4 ? 2 : 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int s = 0; s < L::q; ++s) {
      mbar_init(&bars->q_full[s], p.q_tma ? 1 : (kFp4 ? 2 : 32));
      mbar_init(&bars->q_empty[s], 1);
      mbar_init(&bars->p_full[s], kSoftmaxThreads);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&bars->s_full[w], 1);
      mbar_init(&bars->s_free[w], kSoftmaxThreads);
      mbar_init(&bars->o_full[w], 1);
      mbar_init(&bars->o_free[w], kSoftmaxThreads);
    }
    for (int m = 0; m < kMetaSlots; ++m) {
      mbar_init(&bars->meta_full[m], kSoftmaxThreads);
      mbar_init(&bars->meta_free[m], kSoftmaxThreads);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if constexpr (kFp4) nvfp4_build_lut(smem + L::off_lut, threadIdx.x, kThreads);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // Launched with 128 registers per thread (512 threads); each role's
  // warpgroup then resizes: softmax 176, epilogue 96, control warps 64
  // (4*32*64 + 8*32*176 + 4*32*96 = 65536).  The softmax needs its 176: at
  // 168 the compiler fits the same code without spills but schedules the
  // exponentials with far less overlap, and the softmax takes twice as long.

  // The five warp roles.  Each lambda runs in exactly one branch of the
  // dispatch below, and the two instantiations call them in different
  // orders.  The order sets where each role's loops lie in the instruction
  // stream, and the roles' hot loops together overflow the instruction
  // caches of an SM sub-partition, so it decides how long warps stall on
  // instruction fetch (ncu: 1.60 such stalls per issue in one layout, 0.92
  // in another, for the same 47.9 M instructions).  The orders below are the
  // fastest of those measured on GB300 among the admissible ones: the four
  // control warps form one warpgroup, and setmaxnreg must be one instruction
  // executed by all warps of a warpgroup, so they share one resize and stay
  // together in the order.  E4M3 pool: softmax, epilogue, then warps 2-3,
  // producer, MMA issuer (attention on long_prefill_1m 116.8 us; 125.1 us
  // with the control warps first, 134 us with the MMA issuer leading them).
  // NVFP4 pool: softmax, epilogue, then producer, warps 2-3 (the V
  // converter), MMA issuer (228.5 us; 231.1 us control warps first).
  auto role_producer = [&]() {
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
    int4* shdr = reinterpret_cast<int4*>(smem + L::off_stage);
    int* stok = reinterpret_cast<int*>(smem + L::off_stage + kStageHdr);
    const uint64_t pol_stream = l2_policy_evict_first();
    const uint64_t pol_keep = l2_policy_evict_last();
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
      const int buf = (base / kBatch) & 1;
      if (base + kBatch < cnt) load_batch(base + kBatch, buf ^ 1);
      for (int j = 0; j < kBatch && base + j < cnt; ++j) {
        const int li = base + j;
        const int ks = li % L::k, vs = li % L::v, qs = li % L::q, rs = li % L::rec;
        const int4 hdr = shdr[buf * kBatch + j];
        const int tok = (lane < 16) ? stok[(buf * kBatch + j) * 16 + lane] : 0;
        int ok = 1;
        if (lane == 0) {
          // NVFP4: the K and V slots of item li - kraw / li - vraw are
          // converted, which also frees record slot li - rec
          if constexpr (kFp4) {
            if (li >= L::kraw)
              ok = bounded_wait(&bars->kraw_empty[li % L::kraw],
                                ((li / L::kraw) - 1) & 1, abort, p.wait_ns);
            if (ok && li >= L::vraw)
              ok = bounded_wait(&bars->vraw_empty[li % L::vraw],
                                ((li / L::vraw) - 1) & 1, abort, p.wait_ns);
          } else {
            // the K tile of item li - k is free once its QK is done, the V
            // tile (and the record slot, rec == v) of item li - v once its PV
            // is done
            if (li >= L::k)
              ok = bounded_wait(&bars->k_empty[ks], ((li / L::k) - 1) & 1,
                                abort, p.wait_ns);
            if (ok && li >= L::v)
              ok = bounded_wait(&bars->v_empty[vs], ((li / L::v) - 1) & 1,
                                abort, p.wait_ns);
          }
          if (ok && li >= L::q)
            ok = bounded_wait(&bars->q_empty[qs], ((li / L::q) - 1) & 1,
                              abort, p.wait_ns);
          if (!ok && !*abort) set_timeout(bars, p.status);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          ok_all = false;
          break;
        }
        if (lane == 0) {
          const uint32_t rec_bytes = 16u * (1u + (uint32_t)hdr.y);
          mbar_arrive_expect_tx(&bars->rec_full[rs], rec_bytes);
          bulk_load(smem + L::off_rec + rs * kRecMax,
                    grec + li * rec_step, rec_bytes,
                    &bars->rec_full[rs]);
          if constexpr (kFp4) {
            const uint8_t* ph = p.kv4 + (int64_t)(hdr.x >> 7) * kFp4PageHead;
            const int kr = li % L::kraw, vr = li % L::vraw;
            mbar_arrive_expect_tx(&bars->kraw_full[kr], kFp4Slot);
            bulk_load(smem + L::off_kraw + kr * kFp4Slot, ph, kFp4Slot,
                      &bars->kraw_full[kr]);
            mbar_arrive_expect_tx(&bars->vraw_full[vr], kFp4Slot);
            bulk_load(smem + L::off_vraw + vr * kFp4Slot, ph + kFp4Slot, kFp4Slot,
                      &bars->vraw_full[vr]);
          } else {
            mbar_arrive_expect_tx(&bars->k_full[ks], kTile);
            tma_load_2d_hint(smem + L::off_k + ks * kTile, &kv_map, &bars->k_full[ks],
                             0, hdr.x, pol_stream);
            mbar_arrive_expect_tx(&bars->v_full[vs], kTile);
            tma_load_2d_hint(smem + L::off_v + vs * kTile, &kv_map, &bars->v_full[vs],
                             kD, hdr.x, pol_stream);
          }
          if (p.q_tma)
            mbar_arrive_expect_tx(&bars->q_full[qs], (uint32_t)(hdr.y * p.G * 128));
        }
        if (p.q_tma) {
          __syncwarp();
          if (lane < hdr.y) {
            void* qdst = smem + L::off_q + qs * kTile +
                         ((lane * p.G + row_rotation(li, p.rotate)) & (kTileM - 1)) * 128;
            tma_load_2d_hint(qdst, &q_map, &bars->q_full[qs], 0, tok * p.Hq + hdr.w,
                             pol_keep);
          }
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
      for (int li = issued > L::rec ? issued - L::rec : 0; li < issued; ++li)
        bounded_wait(&bars->rec_full[li % L::rec], (li / L::rec) & 1,
                     nullptr, kWaitLimitNs);
      if constexpr (kFp4) {
        for (int li = issued > L::kraw ? issued - L::kraw : 0; li < issued; ++li)
          bounded_wait(&bars->kraw_full[li % L::kraw], (li / L::kraw) & 1,
                       nullptr, kWaitLimitNs);
        for (int li = issued > L::vraw ? issued - L::vraw : 0; li < issued; ++li)
          bounded_wait(&bars->vraw_full[li % L::vraw], (li / L::vraw) & 1,
                       nullptr, kWaitLimitNs);
      } else {
        for (int li = issued > L::k ? issued - L::k : 0; li < issued; ++li)
          bounded_wait(&bars->k_full[li % L::k], (li / L::k) & 1,
                       nullptr, kWaitLimitNs);
        for (int li = issued > L::v ? issued - L::v : 0; li < issued; ++li)
          bounded_wait(&bars->v_full[li % L::v], (li / L::v) & 1,
                       nullptr, kWaitLimitNs);
      }
      if (p.q_tma)
        for (int li = issued > L::q ? issued - L::q : 0; li < issued; ++li)
          bounded_wait(&bars->q_full[li % L::q], (li / L::q) & 1,
                       nullptr, kWaitLimitNs);
    }
    __syncwarp();
  };
  auto role_mma = [&]() {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_e4m3_f32(128, 128, false);
      constexpr uint32_t idesc_pv = idesc_e4m3_f32(128, 128, true);
      bool ok = true;
      auto issue_qk = [&](int li) {
        const int ks = li % L::k, qs = li % L::q, w = li & 1;
        tc_fence_after();
        const uint64_t a = smem_desc_sw128(smem_u32(smem + L::off_q + qs * kTile), 16, 1024);
        const uint64_t b = smem_desc_sw128(smem_u32(smem + L::off_k + ks * kTile), 16, 1024);
        const uint32_t d = tmem + (uint32_t)(w * 256);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // K = 128 bytes = 4 x 32
          mma_f8f6f4(d, a + (uint64_t)(kk * 2), b + (uint64_t)(kk * 2), idesc_qk,
                     kk > 0);
        mma_commit(&bars->s_full[w]);
        mma_commit(&bars->k_empty[ks]);
      };
      auto issue_pv = [&](int li) {
        const int vs = li % L::v, qs = li % L::q, w = li & 1;
        tc_fence_after();
        const uint64_t a = smem_desc_sw128(smem_u32(smem + L::off_q + qs * kTile), 16, 1024);
        const uint64_t b = smem_desc_sw128(smem_u32(smem + L::off_v + vs * kTile), 1024, 1024);
        const uint32_t d = tmem + (uint32_t)(w * 256 + 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 128 keys = 4 x 32; V rows advance 4 KB
          mma_f8f6f4(d, a + (uint64_t)(kk * 2), b + (uint64_t)(kk * 256),
                     idesc_pv, kk > 0);
        mma_commit(&bars->o_full[w]);
        mma_commit(&bars->v_empty[vs]);
        mma_commit(&bars->q_empty[qs]);
      };
      // in-order issue of QK(qk) and PV(pv), each as soon as it is ready;
      // QK(n) reuses the S tile of item n-2, free once the softmax has
      // loaded S(n-2) into registers
      int qk = 0, pv = 0;
      uint32_t idle_since = (uint32_t)global_timer_ns();
      while (pv < cnt) {
        bool progressed = false;
        if (qk < cnt) {
          const int k = qk >> 1;
          if ((k == 0 || mbar_test(&bars->s_free[qk & 1], (k - 1) & 1)) &&
              mbar_test(&bars->k_full[qk % L::k], (qk / L::k) & 1) &&
              mbar_test(&bars->q_full[qk % L::q], (qk / L::q) & 1)) {
            issue_qk(qk);
            ++qk;
            progressed = true;
          }
        }
        if (pv < qk) {
          const int w = pv & 1, k = pv >> 1;
          if (mbar_test(&bars->p_full[pv % L::q], (pv / L::q) & 1) &&
              (k == 0 || mbar_test(&bars->o_free[w], (k - 1) & 1)) &&
              mbar_test(&bars->v_full[pv % L::v], (pv / L::v) & 1)) {
            issue_pv(pv);
            ++pv;
            progressed = true;
          }
        }
        if (progressed) {
          idle_since = (uint32_t)global_timer_ns();
        } else if (*abort || (uint32_t)global_timer_ns() - idle_since > p.wait_ns) {
          ok = false;
          break;
        }
      }
      if (!ok && !*abort) set_timeout(bars, p.status);
      mma_commit(&bars->mma_done);
      bounded_wait(&bars->mma_done, 0, nullptr, kWaitLimitNs);
    }
  };
  auto role_warps23 = [&]() {
    // Q rows of item li (cp.async mode): 16-byte chunks into the
    // 128-byte-swizzled K-major tile, `nthr` threads from thread `tid`
    auto gather_q = [&](int li, int tid, int nthr) {
      const int4* rec =
          reinterpret_cast<const int4*>(smem + L::off_rec + (li % L::rec) * kRecMax);
      const int4 hdr = rec[0];
      const int rows = hdr.y * p.G;
      const int rot = row_rotation(li, p.rotate);
      const uint32_t dst0 = smem_u32(smem + L::off_q + (li % L::q) * kTile);
      for (int e = tid; e < rows * 8; e += nthr) {
        const int lrow = e >> 3, ch = e & 7;
        const int i = div_G(lrow, p.inv_G), g = lrow - i * p.G;
        const int row = (lrow + rot) & (kTileM - 1);
        const int t = rec[1 + i].x;
        const uint8_t* src = p.q + ((int64_t)t * p.Hq + hdr.w + g) * kD + ch * 16;
        cp_async_16(dst0 + row * 128 + ((ch ^ (row & 7)) << 4), src);
      }
      cp_async_commit();
    };
    auto wait_rec_q = [&](int li) {
      return warp_wait(&bars->rec_full[li % L::rec], (li / L::rec) & 1, abort,
                          p.wait_ns) &&
             (li < L::q || warp_wait(&bars->q_empty[li % L::q],
                                        ((li / L::q) - 1) & 1, abort, p.wait_ns));
    };
    if constexpr (kFp4) {
      // ---------------------------------------------------------- V converter
      // both warps on every item: the Q gather first (cp.async mode), then
      // the V slot once PV of item li - 2 has freed its tile, followed by a
      // proxy fence so the tensor cores see the generic-proxy stores
      const int c = threadIdx.x - 64;
      bool ok = true;
      for (int li = 0; li < cnt; ++li) {
        const int vs = li % L::v, r = li % L::vraw;
        if (!p.q_tma) {
          if (!wait_rec_q(li)) { ok = false; break; }
          gather_q(li, c, 64);
          cp_async_wait<0>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->q_full[li % L::q]);
        }
        if (!warp_wait(&bars->vraw_full[r], (li / L::vraw) & 1, abort, p.wait_ns) ||
            (li >= L::v && !warp_wait(&bars->v_empty[vs], ((li / L::v) - 1) & 1,
                                          abort, p.wait_ns))) {
          ok = false;
          break;
        }
        convert_slot<64>(smem + L::off_vraw + r * kFp4Slot,
                         smem + L::off_v + vs * kTile, smem + L::off_lut, c);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars->v_full[vs]);
          mbar_arrive(&bars->vraw_empty[r]);
        }
      }
      cp_async_wait<0>();
      if (!ok && lane == 0 && !*abort) set_timeout(bars, p.status);
    } else if (!p.q_tma) {
      // ---------------------------------------------------------- Q gather
      // two warps take alternate items; every lane arrives on q_full
      bool ok = true;
      for (int li = warp - 2; li < cnt; li += 2) {
        if (!wait_rec_q(li)) {
          ok = false;
          break;
        }
        gather_q(li, lane, 32);
        cp_async_wait<0>();
        fence_proxy_async_smem();
        mbar_arrive(&bars->q_full[li % L::q]);
      }
      cp_async_wait<0>();
      if (!ok && lane == 0 && !*abort) set_timeout(bars, p.status);
    }
  };
  auto role_softmax = [&]() {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int w = (warp - 4) >> 2;       // group
    const int quad = warp & 3;           // TMEM lane quadrant
    const int row = quad * 32 + lane;    // tile row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + (uint32_t)(w * 256);
    RowMeta* meta = reinterpret_cast<RowMeta*>(smem + L::off_meta);
    // NVFP4: the group dequantises the K slot of each of its items; item j
    // (j >= 2) right after P(j - 2), whose QK has freed the K tile
    auto convert_k = [&](int j) {
      constexpr int R = kFp4 ? L::kraw : 1;  // (E4M3: never called)
      const int ks = j % L::k, r = j % R;
      if (!warp_wait(&bars->kraw_full[r], (j / R) & 1, abort, p.wait_ns) ||
          (j >= L::k && !warp_wait(&bars->k_empty[ks], ((j / L::k) - 1) & 1,
                                       abort, p.wait_ns))) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        return false;
      }
      convert_slot<128>(smem + L::off_kraw + r * kFp4Slot, smem + L::off_k + ks * kTile,
                        smem + L::off_lut, threadIdx.x - 128 - 128 * w);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->k_full[ks]);
        mbar_arrive(&bars->kraw_empty[r]);
      }
      return true;
    };
    bool ok_k = true;
    if constexpr (kFp4) ok_k = w >= cnt || convert_k(w);
    for (int k = 0; ok_k; ++k) {
      const int li = 2 * k + w;
      if (li >= cnt) break;
      const int rs = li % L::rec;
      if (!warp_wait(&bars->rec_full[rs], (li / L::rec) & 1, abort,
                        p.wait_ns)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      const int4* rec = reinterpret_cast<const int4*>(smem + L::off_rec + rs * kRecMax);
      const int4 hdr = rec[0];
      // logical row (token i, head g) held by this lane for this item
      const int lrow = (row - row_rotation(li, p.rotate)) & (kTileM - 1);
      const int i = div_G(lrow, p.inv_G), g = lrow - i * p.G;
      const bool valid = i < hdr.y;
      const bool warp_valid = __any_sync(0xffffffffu, valid);
      int32_t prow = -1;
      int kv_lim = 127;
      if (valid) {
        const int4 tok = rec[1 + i];
        prow = (tok.x * p.Hq + hdr.w + g) * kTopK + tok.z;
        kv_lim = min(tok.y - hdr.z, 127);
      }
      const bool need_mask = __any_sync(0xffffffffu, valid && kv_lim < 127);
      if (!warp_wait(&bars->s_full[w], k & 1, abort, p.wait_ns)) {
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
      // P goes into the item's own Q/P slot: Q is dead once QK has completed
      // (s_full), so nothing here waits for an earlier item's PV
      uint8_t* prow_s = smem + L::off_q + (li % L::q) * kTile + row * 128;
      float m2 = -INFINITY, l = 0.f;
      if (warp_valid) {
        if (need_mask) {
          mask32(r0, 0, kv_lim);
          mask32(r1, 32, kv_lim);
          mask32(r2, 64, kv_lim);
          mask32(r3, 96, kv_lim);
        }
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        max32(r0, mq);
        max32(r1, mq);
        max32(r2, mq);
        max32(r3, mq);
        const float m = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        m2 = m * p.score_log2;
        // p = 2^(x * c - m2 + 8): probabilities scaled by 256 so that small
        // ones stay out of E4M3's subnormal range; l and O carry the same
        // factor, which cancels.
        const float off = (m2 == -INFINITY) ? 0.f : 8.f - m2;
        const float c = p.score_log2;
        float lq[4] = {0.f, 0.f, 0.f, 0.f};
        exp_pack32(r0, 0, c, off, prow_s, row, lq);
        exp_pack32(r1, 32, c, off, prow_s, row, lq);
        exp_pack32(r2, 64, c, off, prow_s, row, lq);
        exp_pack32(r3, 96, c, off, prow_s, row, lq);
        l = (lq[0] + lq[1]) + (lq[2] + lq[3]);
      }
      // the row-meta slot is free once the epilogue has read item li - 4's
      if (li >= kMetaSlots &&
          !warp_wait(&bars->meta_free[li % kMetaSlots], ((li / kMetaSlots) - 1) & 1,
                        abort, p.wait_ns)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      RowMeta mt;
      mt.prow = prow;
      mt.inv = l > 0.f ? 1.f / l : 0.f;  // O in V's code units; the combine scales
      mt.lse = l > 0.f ? (m2 + __log2f(l) - 8.f) * 0.69314718055994530942f
                       : -INFINITY;
      meta[(li % kMetaSlots) * kTileM + row] = mt;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full[li % L::q]);
      mbar_arrive(&bars->meta_full[li % kMetaSlots]);
      if constexpr (kFp4) {
        if (li + 2 < cnt && !convert_k(li + 2)) break;
      }
    }
  };
  auto role_epilogue = [&]() {
    setmaxnreg_dec<kRegsEpilogue>();
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const RowMeta* meta = reinterpret_cast<const RowMeta*>(smem + L::off_meta);
    const uint64_t pol_keep = l2_policy_evict_last();
    for (int li = 0; li < cnt; ++li) {
      const int w = li & 1, k = li >> 1;
      if (!warp_wait(&bars->meta_full[li % kMetaSlots],
                        (li / kMetaSlots) & 1, abort, p.wait_ns)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      const RowMeta mt = meta[(li % kMetaSlots) * kTileM + row];
      mbar_arrive(&bars->meta_free[li % kMetaSlots]);
      const bool valid = mt.prow >= 0;
      const bool warp_valid = __any_sync(0xffffffffu, valid);
      if (!warp_wait(&bars->o_full[w], k & 1, abort, p.wait_ns)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      tc_fence_after();
      if (warp_valid) {
        const uint32_t o_tmem = tmem + lane_off + (uint32_t)(w * 256 + 128);
        uint8_t* dst = p.part_o + mt.prow * (int64_t)kD;
        // one half per iteration, the loop kept rolled: the instruction
        // cache is shared with the other warp roles' loops
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t ra[32], rb[32];
          __syncwarp();
          tmem_ld32(o_tmem + half * 64, ra);
          tmem_ld32(o_tmem + half * 64 + 32, rb);
          tmem_wait_ld();
          if (valid)
            store_partial_half(ra, rb, mt.inv, dst + half * 64,
                               p.part_big + mt.prow * (int64_t)(2 * kD) + half * 128,
                               p.e4m3_over4, pol_keep);
        }
        if (valid) st_global_f32_hint(p.part_lse + mt.prow, mt.lse, pol_keep);
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free[w]);
    }
  };
  if constexpr (kFp4) {
    if (warp >= 4 && warp < 12) {
      role_softmax();
    } else if (warp >= 12) {
      role_epilogue();
    } else {
      setmaxnreg_dec<kRegsControl>();
      if (warp == 0) role_producer();
      else if (warp >= 2) role_warps23();
      else role_mma();
    }
  } else {
    if (warp >= 4 && warp < 12) {
      role_softmax();
    } else if (warp >= 12) {
      role_epilogue();
    } else {
      setmaxnreg_dec<kRegsControl>();
      if (warp >= 2) role_warps23();
      else if (warp == 0) role_producer();
      else role_mma();
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

// The dynamic shared-memory limit is a per-device function attribute: set
// it once for every device the kernel is launched on.
template <bool kFp4, int kDepth>
cudaError_t launch_kernel(const CUtensorMap& kv_map, const CUtensorMap& q_map,
                          const Params& p, int64_t grid, cudaStream_t stream) {
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> attr_set[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(attention_kernel<kFp4, kDepth>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Ring<kFp4, kDepth>::bytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_set[dev].store(true, std::memory_order_release);
  }
  return launch_pdl(attention_kernel<kFp4, kDepth>, dim3((unsigned)grid), dim3(kThreads),
                    Ring<kFp4, kDepth>::bytes, stream, kv_map, q_map, p);
}

}  // namespace

uint32_t partial_over4(float v_scale) {
  // value of a non-negative E4M3 code 0x00 .. 0x7E (OCP E4M3: bias 7,
  // subnormals m * 2^-9)
  auto value = [](uint32_t c) {
    const int e = (int)(c >> 3), m = (int)(c & 7);
    return e == 0 ? std::ldexp((double)m, -9) : std::ldexp(1.0 + m / 8.0, e - 7);
  };
  const double lim = (double)kE4M3PartialLimit / (double)v_scale;
  uint32_t c = 0;
  while (c < 0x7E && value(c + 1) <= lim) ++c;
  if (lim >= 448.0) c = 0x7F;
  return (0x7Fu - c) * 0x01010101u;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  const msa_plan_t& pl = *a.plan;
  if (pl.max_work == 0) return cudaSuccess;
  if (a.q_bf16) return launch_attention_bf16q(a, stream);
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int G = (int)(pl.Hq / pl.Hkv);
  const bool fp4 = a.kv_format == MSA_KV_NVFP4;
  // E4M3 page pool: rows = (page, KV head, token), 256 bytes each (K then
  // V).  An NVFP4 pool is read by plain bulk copies, with no tensor map.
  CUtensorMap kv_map, q_map;
  memset(&kv_map, 0, sizeof(kv_map));
  memset(&q_map, 0, sizeof(q_map));
  if (!fp4 && !encode_rows(enc, &kv_map, a.kv, 2 * kD,
                           (uint64_t)a.num_pages * pl.Hkv * kPage, 128))
    return cudaErrorInvalidValue;
  // queries: rows = (token, query head), 128 bytes each; one box = the G
  // heads of one KV head of one token
  const bool q_tma = (G % 8) == 0;
  if (q_tma) {
    if (!encode_rows(enc, &q_map, a.q, kD, (uint64_t)pl.T * pl.Hq, (uint32_t)G))
      return cudaErrorInvalidValue;
  }

  Params p;
  p.q = a.q;
  p.kv4 = fp4 ? a.kv : nullptr;
  p.records = reinterpret_cast<const int4*>(pl.records);
  p.rec_stride = (int)(pl.record_bytes / 16);
  p.counters = pl.counters;
  p.part_o = a.part_o;
  p.part_vscale = a.part_vscale;
  p.part_lse = a.part_lse;
  p.part_big = a.part_big;
  p.e4m3_over4 = partial_over4(a.v_scale);
  p.status = pl.status;
  p.Hq = (int)pl.Hq;
  p.G = G;
  p.rotate = (G <= 32 && 32 % G == 0) ? 1 : 0;
  p.inv_G = 1.0f / (float)G;
  p.q_tma = q_tma ? 1 : 0;
  p.score_log2 = a.score_log2;
  p.v_scale = a.v_scale;
  p.wait_ns = (uint32_t)std::min<uint64_t>(pipeline_wait_limit_ns(), kWaitLimitNs);

  const int64_t grid = std::min<int64_t>(num_sms(), pl.max_work);
  if (fp4) return launch_kernel<true, 5>(kv_map, q_map, p, grid, stream);
  return plan_is_sparse(pl.rows, pl.bitmap_words, pl.T, pl.Hkv)
             ? launch_kernel<false, 5>(kv_map, q_map, p, grid, stream)
             : launch_kernel<false, 3>(kv_map, q_map, p, grid, stream);
}

}  // namespace msa
