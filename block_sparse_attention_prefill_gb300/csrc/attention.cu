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
// One CTA per SM, persistent over a contiguous range of the work list.
// Every work item has a record written by the plan: {KV row of the page in
// the pool, token count n, first key position, first query head} and, per
// token, {token id, query position, top-k slot}.  Warp roles (16 warps):
//   warp 0      producer: bulk copy of the item's record, TMA loads of the
//               K and V halves of the page (2 x 16 KB, 128-byte swizzle)
//               and, when G is a multiple of 8, of the Q rows: one box of G
//               rows per token, issued by one lane per token from token ids
//               prefetched out of the record in global memory
//   warp 1      tcgen05 issuer (one thread) and TMEM owner (512 columns)
//   warps 2-3   Q gather when G is not a multiple of 8: cp.async of 16-byte
//               chunks into the 128-byte-swizzled K-major tile
//   warps 4-7   softmax group 0 (even items)
//   warps 8-11  softmax group 1 (odd items)
//   warps 12-15 epilogue: O from TMEM, normalised, bf16 partials to HBM
// Shared memory: a 4-slot ring of {K, V} 16 KB tiles with the item's record
// (released when PV completes), a 3-slot ring of Q tiles (released when QK
// completes), 2 P tiles, and a 4-slot ring of per-row results handed from
// softmax to epilogue.
// TMEM: per group an S tile (128 columns) and an O tile (128 columns).
// The MMA thread issues QK(n) and PV(n) as soon as each one's inputs are
// ready, in order, so the tensor cores compute item n+1's scores while item
// n's softmax runs and never wait on one item for the next one's data.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kKvStages = 4;
constexpr int kQStages = 3;
constexpr int kBatch = 8;  // items whose headers / token ids are prefetched
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
constexpr int kOffBar = kOffMeta + kMetaSlots * kTileM * (int)sizeof(RowMeta);

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
  uint16_t* part_o;
  float* part_lse;
  uint32_t* status;
  int Hq, G;
  int q_tma;       // 1: Q rows by TMA (G % 8 == 0), 0: by cp.async
  float score_log2;
  float v_scale;
};

__device__ __forceinline__ void set_timeout(Barriers* bars, uint32_t* status) {
  bars->abort = 1;
  atomicOr(status, (unsigned)MSA_STATUS_TIMEOUT);
}

// Where the rows (token i, query head g) of an item sit in the 128-row tile.
// When G divides 32 the tokens are dealt round-robin over the four TMEM lane
// quadrants (token i -> quadrant i % 4, G consecutive lanes), so that even a
// small item keeps all four warps of a softmax group -- and all four SM
// sub-partitions -- busy; otherwise tokens take consecutive rows.  Either
// way a token's G rows are consecutive and start at a multiple of G, which
// is what one TMA box of G rows needs.
__device__ __forceinline__ int tile_row(int i, int g, int G) {
  return (32 % G == 0) ? 32 * (i & 3) + (i >> 2) * G + g : i * G + g;
}
__device__ __forceinline__ void row_token(int q, int ql, int G, int& i, int& g) {
  if (32 % G == 0) {
    i = q + 4 * (ql / G);
    g = ql % G;
  } else {
    const int r = 32 * q + ql;
    i = r / G;
    g = r % G;
  }
}
// rows of quadrant q that hold queries of an n-token item: [0, result)
__device__ __forceinline__ int quad_rows(int q, int n, int G) {
  if (32 % G == 0) return (n > q ? (n - q + 3) >> 2 : 0) * G;
  const int r = n * G - 32 * q;
  return r < 0 ? 0 : (r > 32 ? 32 : r);
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Row maximum over a thread's 32 columns of one row in a 16x256b fragment
// (registers 4i + sel, 4i + sel + 1 for column block i), then over the four
// threads that share the row.  Columns past kv_lim are masked when kMask.
template <bool kMask>
__device__ __forceinline__ float frag_row_max(const uint32_t (&v)[64], int sel,
                                              int tc, int kv_lim) {
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float x0 = __uint_as_float(v[4 * i + sel]);
    float x1 = __uint_as_float(v[4 * i + sel + 1]);
    if (kMask) {
      const int c = 8 * i + 2 * tc;
      if (c > kv_lim) x0 = -INFINITY;
      if (c + 1 > kv_lim) x1 = -INFINITY;
    }
    m = max3f(m, x0, x1);
  }
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  return m;
}

// p = 2^(x * c + off) for the thread's 32 columns of one row, rounded to
// E4M3 in pairs and stored into the 128-byte-swizzled P row `trow`; returns
// the row sum over the four threads of the row.
template <bool kMask>
__device__ __forceinline__ float frag_row_exp(const uint32_t (&v)[64], int sel,
                                              int tc, int kv_lim, float c,
                                              float off, uint8_t* sP,
                                              int trow) {
  float l = 0.f;
  uint8_t* prow = sP + trow * 128 + 2 * tc;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float p0 = ex2_approx(fmaf(__uint_as_float(v[4 * i + sel]), c, off));
    float p1 = ex2_approx(fmaf(__uint_as_float(v[4 * i + sel + 1]), c, off));
    if (kMask) {
      const int col = 8 * i + 2 * tc;
      if (col > kv_lim) p0 = 0.f;
      if (col + 1 > kv_lim) p1 = 0.f;
    }
    l += p0 + p1;
    const uint16_t e = __nv_cvt_float2_to_fp8x2(make_float2(p0, p1),
                                                __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<uint16_t*>(prow + ((((i >> 1) ^ (trow & 7))) << 4) +
                                 8 * (i & 1)) = e;
  }
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  return l;
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

  const int num_work = p.counters[1];
  const int begin = (int)((int64_t)blockIdx.x * num_work / gridDim.x);
  const int end = (int)((int64_t)(blockIdx.x + 1) * num_work / gridDim.x);
  const int cnt = end - begin;

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
  // warpgroup then resizes: softmax 176, epilogue 96, control warps 64
  // (4*32*64 + 8*32*176 + 4*32*96 = 65536).

  if (warp < 4) {
  setmaxnreg_dec<kRegsControl>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // lane 0 waits for a free K|V slot and issues the record / K / V copies.
    // Headers are prefetched kBatch items ahead: lane j of the warp holds
    // the header of item base + j of the current batch and of the next one.
    const int4* grec = p.records + (int64_t)begin * p.rec_stride;
    int4 hcur = make_int4(0, 0, 0, 0), hnext = make_int4(0, 0, 0, 0);
    if (lane < kBatch && lane < cnt) hcur = grec[(int64_t)lane * p.rec_stride];
    int issued = 0;
    bool ok = true;
    for (int base = 0; ok && base < cnt; base += kBatch) {
      if (lane < kBatch && base + kBatch + lane < cnt)
        hnext = grec[(int64_t)(base + kBatch + lane) * p.rec_stride];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int li = base + j;
        if (li >= cnt) break;
        const int4 hdr = make_int4(__shfl_sync(0xffffffffu, hcur.x, j),
                                   __shfl_sync(0xffffffffu, hcur.y, j), 0, 0);
        const int ks = li % kKvStages;
        if (lane == 0) {
          int w_ok = 1;
          if (li >= kKvStages)
            w_ok = bounded_wait(&bars->kv_empty[ks], ((li / kKvStages) - 1) & 1,
                                abort, kWaitLimitNs);
          if (w_ok) {
            const uint32_t rec_bytes = 16u * (1u + (uint32_t)hdr.y);
            mbar_arrive_expect_tx(&bars->rec_full[ks], rec_bytes);
            bulk_load(smem + kOffRec + ks * kRecMax,
                      p.records + (int64_t)(begin + li) * p.rec_stride,
                      rec_bytes, &bars->rec_full[ks]);
            mbar_arrive_expect_tx(&bars->kv_full[ks], 2 * kTile);
            tma_load_2d(smem + kOffK + ks * kTile, &kv_map, &bars->kv_full[ks], 0, hdr.x);
            tma_load_2d(smem + kOffV + ks * kTile, &kv_map, &bars->kv_full[ks], kD, hdr.x);
            issued = li + 1;
          } else if (!*abort) {
            set_timeout(bars, p.status);
          }
          ok = w_ok;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      hcur = hnext;
    }
    // every copy this warp started must land before the CTA exits
    if (lane == 0)
      for (int li = issued > kKvStages ? issued - kKvStages : 0; li < issued; ++li) {
        bounded_wait(&bars->rec_full[li % kKvStages], (li / kKvStages) & 1,
                     nullptr, kWaitLimitNs);
        bounded_wait(&bars->kv_full[li % kKvStages], (li / kKvStages) & 1,
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
      // QK(n) reuses the S tile of item n-2, free once the softmax warps
      // have read it into registers (s_free)
      int qk = 0, pv = 0;
      uint64_t idle_since = global_timer_ns();
      while (pv < cnt) {
        bool progressed = false;
        if (qk < cnt &&
            (qk < 2 || mbar_test(&bars->s_free[qk & 1], ((qk >> 1) - 1) & 1))) {
          if (mbar_test(&bars->kv_full[qk % kKvStages], (qk / kKvStages) & 1) &&
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
        } else {
          // nothing ready: yield the issue slots to the softmax warps that
          // share this SM sub-partition
          __nanosleep(64);
        }
      }
      if (!ok && !*abort) set_timeout(bars, p.status);
      mma_commit(&bars->mma_done);
      bounded_wait(&bars->mma_done, 0, nullptr, kWaitLimitNs);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ Q gather
    if (p.q_tma) {
      // warp 2: one TMA box of G rows per token, lane i issues token i
      // (C = 128 / G <= 16).  Token ids and headers are prefetched kBatch
      // items ahead from the records in global memory: lane i < C holds
      // token i of each item of the batch, lane j < kBatch the header of
      // item base + j.
      if (warp == 2) {
        const int4* grec = p.records + (int64_t)begin * p.rec_stride;
        const int C = kTileM / p.G;
        int tcur[kBatch], tnext[kBatch];
        int4 hcur = make_int4(0, 0, 0, 0), hnext = make_int4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          tcur[j] = (j < cnt && lane < C) ? grec[(int64_t)j * p.rec_stride + 1 + lane].x : 0;
          tnext[j] = 0;
        }
        if (lane < kBatch && lane < cnt) hcur = grec[(int64_t)lane * p.rec_stride];
        int issued = 0;
        bool ok = true;
        for (int base = 0; ok && base < cnt; base += kBatch) {
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int li = base + kBatch + j;
            if (li < cnt && lane < C)
              tnext[j] = grec[(int64_t)li * p.rec_stride + 1 + lane].x;
          }
          if (lane < kBatch && base + kBatch + lane < cnt)
            hnext = grec[(int64_t)(base + kBatch + lane) * p.rec_stride];
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int li = base + j;
            if (li >= cnt) break;
            const int n = __shfl_sync(0xffffffffu, hcur.y, j);
            const int hq0 = __shfl_sync(0xffffffffu, hcur.w, j);
            const int qs = li % kQStages;
            if (lane == 0) {
              int w_ok = 1;
              if (li >= kQStages)
                w_ok = bounded_wait(&bars->q_empty[qs], ((li / kQStages) - 1) & 1,
                                    abort, kWaitLimitNs);
              if (w_ok)
                mbar_arrive_expect_tx(&bars->q_full[qs], (uint32_t)(n * p.G * 128));
              else if (!*abort)
                set_timeout(bars, p.status);
              ok = w_ok;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane < n)
              tma_load_2d(smem + kOffQ + qs * kTile + tile_row(lane, 0, p.G) * 128,
                          &q_map, &bars->q_full[qs], 0, tcur[j] * p.Hq + hq0);
            issued = li + 1;
          }
#pragma unroll
          for (int j = 0; j < kBatch; ++j) tcur[j] = tnext[j];
          hcur = hnext;
        }
        if (lane == 0)
          for (int li = issued > kQStages ? issued - kQStages : 0; li < issued; ++li)
            bounded_wait(&bars->q_full[li % kQStages], (li / kQStages) & 1,
                         nullptr, kWaitLimitNs);
        __syncwarp();
      }
    }
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
        const uint32_t dst0 = smem_u32(smem + kOffQ + qs * kTile);
        for (int e = lane; e < rows * 8; e += 32) {
          const int lrow = e >> 3, ch = e & 7;
          const int i = lrow / p.G, g = lrow - i * p.G;
          const int row = tile_row(i, g, p.G);
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
    // Warp `quad` of group w owns TMEM lanes 32*quad .. +31 (tile rows).  It
    // reads S with the 16x256b shape: thread t holds, per 16-lane half, rows
    // t/4 and t/4 + 8 at columns 8i + 2(t%4) + {0,1}, so four threads share a
    // row and a quadrant with 8 query rows costs each thread 32 columns.
    const int w = (warp - 4) >> 2;       // group
    const int quad = warp & 3;           // TMEM lane quadrant
    const int t4 = lane >> 2, tc = lane & 3;
    const uint32_t s_tmem = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(w * 256);
    uint8_t* sP = smem + kOffP + w * kTile;
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
      const int R = quad_rows(quad, hdr.y, p.G);
      const int nh = (R + 15) >> 4;      // 16-lane halves holding rows
      // my rows: r = 2h + b -> quadrant row 16h + t4 + 8b
      int64_t prow[4];
      int kvl[4];
      bool any_mask = false;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int ql = 16 * (r >> 1) + t4 + 8 * (r & 1);
        prow[r] = -1;
        kvl[r] = 127;
        if (ql < R) {
          int i, g;
          row_token(quad, ql, p.G, i, g);
          const int4 tok = rec[1 + i];
          prow[r] = ((int64_t)tok.x * p.Hq + hdr.w + g) * kTopK + tok.z;
          kvl[r] = min(tok.y - hdr.z, 127);
          any_mask |= kvl[r] < 127;
        }
      }
      const bool need_mask = __any_sync(0xffffffffu, any_mask);
      if (!bounded_wait(&bars->s_full[w], k & 1, abort, kWaitLimitNs)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      tc_fence_after();
      const float c = p.score_log2;
      float m2[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      float l[4] = {0.f, 0.f, 0.f, 0.f};
      bool p_free = true;
      if (nh == 0) {
        mbar_arrive(&bars->s_free[w]);
      } else {
        __syncwarp();
        uint32_t v0[64], v1[64];
        tmem_ld_16x256b_x16(s_tmem, v0);
        if (nh > 1) tmem_ld_16x256b_x16(s_tmem + (16u << 16), v1);
        tmem_wait_ld();
        // S is in registers: the tile can take the next item's scores
        tc_fence_before();
        mbar_arrive(&bars->s_free[w]);
        float m[4];
        if (need_mask) {
          m[0] = frag_row_max<true>(v0, 0, tc, kvl[0]);
          m[1] = frag_row_max<true>(v0, 2, tc, kvl[1]);
          if (nh > 1) {
            m[2] = frag_row_max<true>(v1, 0, tc, kvl[2]);
            m[3] = frag_row_max<true>(v1, 2, tc, kvl[3]);
          }
        } else {
          m[0] = frag_row_max<false>(v0, 0, tc, 127);
          m[1] = frag_row_max<false>(v0, 2, tc, 127);
          if (nh > 1) {
            m[2] = frag_row_max<false>(v1, 0, tc, 127);
            m[3] = frag_row_max<false>(v1, 2, tc, 127);
          }
        }
        // p = 2^(x * c - m2 + 8): probabilities scaled by 256 so that small
        // ones stay out of E4M3's subnormal range; l and O carry the same
        // factor, which cancels.
        float off[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          m2[r] = (r < 2 * nh) ? m[r] * c : -INFINITY;
          off[r] = (m2[r] == -INFINITY) ? 0.f : 8.f - m2[r];
        }
        // the P tile is free once PV of this group's previous item is done
        if (k > 0)
          p_free = bounded_wait(&bars->o_full[w], (k - 1) & 1, abort, kWaitLimitNs);
        if (p_free) {
          const int row0 = 32 * quad + t4;
          if (need_mask) {
            l[0] = frag_row_exp<true>(v0, 0, tc, kvl[0], c, off[0], sP, row0);
            if (R > 8) l[1] = frag_row_exp<true>(v0, 2, tc, kvl[1], c, off[1], sP, row0 + 8);
            if (nh > 1) {
              l[2] = frag_row_exp<true>(v1, 0, tc, kvl[2], c, off[2], sP, row0 + 16);
              if (R > 24) l[3] = frag_row_exp<true>(v1, 2, tc, kvl[3], c, off[3], sP, row0 + 24);
            }
          } else {
            l[0] = frag_row_exp<false>(v0, 0, tc, 127, c, off[0], sP, row0);
            if (R > 8) l[1] = frag_row_exp<false>(v0, 2, tc, 127, c, off[1], sP, row0 + 8);
            if (nh > 1) {
              l[2] = frag_row_exp<false>(v1, 0, tc, 127, c, off[2], sP, row0 + 16);
              if (R > 24) l[3] = frag_row_exp<false>(v1, 2, tc, 127, c, off[3], sP, row0 + 24);
            }
          }
        }
      }
      // Every thread, with or without rows, waits for PV of item li-2 before
      // it writes the result ring: that PV needed the epilogue of item li-4,
      // the last reader of this ring slot, to be done.
      if (nh == 0 && k > 0)
        p_free = bounded_wait(&bars->o_full[w], (k - 1) & 1, abort, kWaitLimitNs);
      if (!p_free) {
        if (!*abort) set_timeout(bars, p.status);
        break;
      }
      if (tc == 0) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          RowMeta mt;
          mt.prow = prow[r];
          mt.inv = l[r] > 0.f ? p.v_scale / l[r] : 0.f;
          mt.lse = l[r] > 0.f
                       ? (m2[r] + __log2f(l[r]) - 8.f) * 0.69314718055994530942f
                       : -INFINITY;
          meta[(li % kMetaSlots) * kTileM + 32 * quad + 16 * (r >> 1) + t4 +
               8 * (r & 1)] = mt;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full[w]);
      mbar_arrive(&bars->meta_full[li % kMetaSlots]);
    }
  } else {
    setmaxnreg_dec<kRegsEpilogue>();
    // ------------------------------------------------------------ epilogue
    // Same 16x256b fragments as the softmax: thread t writes columns
    // 8i + 2(t%4) + {0,1} of rows t/4 (+8, +16, +24) of its quadrant.
    const int quad = warp & 3;
    const int t4 = lane >> 2, tc = lane & 3;
    const RowMeta* meta = reinterpret_cast<const RowMeta*>(smem + kOffMeta);
    for (int li = 0; li < cnt; ++li) {
      const int w = li & 1, k = li >> 1;
      if (!bounded_wait(&bars->meta_full[li % kMetaSlots],
                        (li / kMetaSlots) & 1, abort, kWaitLimitNs)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      RowMeta mt[4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
        mt[r] = meta[(li % kMetaSlots) * kTileM + 32 * quad + 16 * (r >> 1) +
                     t4 + 8 * (r & 1)];
      const bool h0 = __any_sync(0xffffffffu, mt[0].prow >= 0 || mt[1].prow >= 0);
      const bool h1 = __any_sync(0xffffffffu, mt[2].prow >= 0 || mt[3].prow >= 0);
      if (!bounded_wait(&bars->o_full[w], k & 1, abort, kWaitLimitNs)) {
        if (lane == 0 && !*abort) set_timeout(bars, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t o_tmem =
          tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(w * 256 + 128);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!(h == 0 ? h0 : h1)) continue;
        uint32_t v[64];
        __syncwarp();
        tmem_ld_16x256b_x16(o_tmem + ((uint32_t)(16 * h) << 16), v);
        tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const RowMeta& m = mt[2 * h + b];
          if (m.prow < 0) continue;
          uint32_t* dst = reinterpret_cast<uint32_t*>(
              p.part_o + m.prow * (int64_t)kD + 2 * tc);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(
                __uint_as_float(v[4 * i + 2 * b]) * m.inv,
                __uint_as_float(v[4 * i + 2 * b + 1]) * m.inv);
            dst[4 * i] = *reinterpret_cast<uint32_t*>(&h2);
          }
          if (tc == 0) p.part_lse[m.prow] = m.lse;
        }
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
  p.part_lse = a.part_lse;
  p.status = pl.status;
  p.Hq = (int)pl.Hq;
  p.G = G;
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
  attention_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(kv_map, q_map, p);
  return cudaGetLastError();
}

}  // namespace msa
