// build_k2q_csr on the device: invert the per-token page lists into
// per-(KV head, page) query lists, plus the work list of the attention
// kernel.  (vLLM docs, sparse_attention_msa, MiniMaxM3SparseMSAImpl.forward:
// build_k2q_csr(topk, cu_seqlens_q, cu_seqlens_k, 128, total_rows =
// total_kv_blocks, qhead_per_kv, return_schedule=True); vLLM PR 60930,
// Details / "Host sync": the plan stays on the device, no host copy.)
//
// Four kernels, all on `stream`, no host synchronisation; each is a
// programmatic dependent launch (its launch overlaps the tail of the kernel
// before it on the stream; on plans whose bitmap is large next to their
// top-k entries, mark and scatter also read, before their wait, what the
// kernels two and more before them produced):
//   prep     CTA 0: per-request row offsets (sum of page counts), checks,
//            status word, counters; every CTA: clears its share of the
//            (row, token) membership bitmap
//   mark     one thread per top-k entry: validate the id, drop repeats, set
//            one bit per kept page in the membership bitmap; the (token,
//            KV head) list's 16 threads together write its slot mask.  This
//            is the histogram, kept as bits: repeats collapse and the order
//            of arrival cannot change the result.
//   rows     one CTA per tile of rows (at most kMaxRowTiles tiles), 1 to 16
//            lanes per row by the row's width: the row's length (popcount of
//            its words), the running count in front of every word, each
//            row's entries and work items in front of it within the tile,
//            and the tile's totals.
//   scatter  every CTA first scans the tiles' totals in shared memory (the
//            exclusive scan across tiles: one load per thread, no waiting
//            on other CTAs) and writes its share of row_ptr; then one thread
//            per top-k entry: each kept entry goes to row_ptr + (tokens of
//            the same row before it), found in O(1) from the word prefix and
//            a popcount, and fills its token slot of the work record the
//            attention kernel will read; the first entry of each chunk also
//            writes the chunk's work item and record header.
// Every output is a function of the inputs alone: bit-exact and
// deterministic run to run.
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kScanThreads = 1024;

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Exclusive scan of one value per thread over a block of kThreads threads;
// every thread receives the block total in *total.
template <int kThreads>
__device__ __forceinline__ int block_excl_scan(int v, int* total) {
  __shared__ int warp_sums[kThreads / 32 + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int incl = warp_incl_scan(v);
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int s = lane < kThreads / 32 ? warp_sums[lane] : 0;
    const int si = warp_incl_scan(s);
    if (lane < kThreads / 32) warp_sums[lane] = si - s;
    if (lane == 31) warp_sums[kThreads / 32] = si;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  *total = warp_sums[kThreads / 32];
  __syncthreads();
  return r;
}

// largest i in [0, n) with a[i] <= x  (a non-decreasing, a[0] <= x)
__device__ __forceinline__ int upper_index(const int32_t* a, int n, int64_t x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct PlanDev {
  const int32_t* topk;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_table;
  int64_t bt_stride, num_pages;
  int B, T, Hkv, G, W, C;
  int early;  // 1: mark and scatter read their inputs before their wait
  int topk_hkv, h_begin;  // topk's KV heads, and the first of this plan's
  int64_t total_rows, rows, max_q, max_k;
  int32_t* req_off;
  uint32_t* bitmap;
  int32_t* word_pre;     // [rows * W] tokens of the row before each word
  int32_t* row_cnt;      // [rows] entries of the row
  int32_t* row_loc;      // [rows][2] entries, work items before the row in its tile
  uint64_t* tile_state;  // [ntiles] tile totals: entries << 32 | work items
  int ntiles, tile_rows, lane_shift;  // rows kernel tiling (see rows)
  int32_t* row_ptr;
  int32_t* q_idx;
  uint8_t* slot;
  int32_t* work;
  int4* records;
  int rec_stride;  // int4 units per record: 1 header + C tokens
  int32_t* counters;
  uint16_t* slot_mask;
  uint32_t* status;
};

// counters[2] == 1 when the per-request metadata passed the checks.
__global__ void __launch_bounds__(kScanThreads) plan_prep_kernel(PlanDev d,
                                                                 int64_t bitmap_vec) {
  // launched as a dependent of whatever kernel ran before it on the stream
  // (the top-k ids may be its output): the launch overlaps that kernel's
  // tail, the work waits for it
  pdl_wait();
  pdl_trigger();
  {
    uint4* bm = reinterpret_cast<uint4*>(d.bitmap);
    const int64_t stride = (int64_t)gridDim.x * kScanThreads;
    const int64_t i0 = (int64_t)blockIdx.x * kScanThreads + threadIdx.x;
    for (int64_t i = i0; i < bitmap_vec; i += stride) bm[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (blockIdx.x != 0) return;
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  bool bad = false, overflow = false;
  if (threadIdx.x == 0) {
    if (d.B > 0 && (d.cu_q[0] != 0 || d.cu_q[d.B] != d.T)) bad = true;
    if (d.B == 0 && d.T != 0) bad = true;
  }
  int carry = 0;
  for (int base = 0; base < d.B; base += kScanThreads) {
    const int b = base + threadIdx.x;
    int pages = 0;
    if (b < d.B) {
      const int64_t ql = (int64_t)d.cu_q[b + 1] - d.cu_q[b];
      const int64_t sl = (int64_t)d.cu_k[b + 1] - d.cu_k[b];
      if (ql < 0 || sl < ql || ql > d.max_q || sl > d.max_k) bad = true;
      else pages = (int)ceil_div(sl, kPage);
    }
    int total;
    const int ex = block_excl_scan<kScanThreads>(pages, &total);
    if (b < d.B) d.req_off[b] = carry + ex;
    carry += total;
    if ((int64_t)carry > d.total_rows) overflow = true;
  }
  if (bad) atomicOr(&s_bad, 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    d.req_off[d.B] = carry;
    unsigned st = 0;
    if (s_bad) st |= MSA_STATUS_BAD_SEQLENS;
    if (!s_bad && overflow) st |= MSA_STATUS_ROWS_OVERFLOW;
    *d.status = st;
    d.counters[2] = st ? 0 : 1;  // the scatter kernel writes [0] and [1]
  }
}

// Element of topk for list w = t * Hkv + h (h among this plan's heads) and
// position j: topk holds topk_hkv heads per token, this plan's from h_begin.
__device__ __forceinline__ int64_t topk_index(const PlanDev& d, int64_t w, int j) {
  if (d.topk_hkv == d.Hkv) return w * kTopK + j;
  const int64_t t = w / d.Hkv;
  return ((t * d.topk_hkv + d.h_begin) + (w - t * d.Hkv)) * kTopK + j;
}

struct TokenInfo {
  int b, i, pos, own, P;
  int64_t row0;
};

// Per-request metadata (cu_seqlens_q, cu_seqlens_k, row offsets), copied
// into shared memory by every CTA of the mark and scatter kernels when the
// batch has fewer than kMetaCache requests, so that a thread's reads of it
// do not add global round trips after its top-k entry; read from global
// memory otherwise.
constexpr int kMetaCache = 512;
struct ReqMeta {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* req_off;
};

// Token t's request, index in it, position, own page and the request's
// page count (m.req_off unused; row0 left 0).
__device__ __forceinline__ TokenInfo token_info_noff(const PlanDev& d, const ReqMeta& m, int t) {
  TokenInfo k;
  k.b = upper_index(m.cu_q, d.B, t);
  k.i = t - m.cu_q[k.b];
  const int64_t ql = m.cu_q[k.b + 1] - m.cu_q[k.b];
  const int64_t sl = m.cu_k[k.b + 1] - m.cu_k[k.b];
  k.pos = (int)(sl - ql + k.i);
  k.own = k.pos / kPage;
  k.P = (int)ceil_div(sl, kPage);
  k.row0 = 0;
  return k;
}

// The same with row0, the CSR row of the token's request's page 0 for KV
// head h.
__device__ __forceinline__ TokenInfo token_info(const PlanDev& d, const ReqMeta& m,
                                                int t, int h) {
  TokenInfo k = token_info_noff(d, m, t);
  k.row0 = (int64_t)h * d.total_rows + m.req_off[k.b];
  return k;
}

// A load before the kernel's dependent-launch wait goes to L2
// (ld.global.cg): only the wait makes earlier kernels' writes visible to
// plain loads.  After the wait, plain loads keep the L1 hits of values that
// many entries share (block_table entries, bitmap words).
template <typename T>
__device__ __forceinline__ T ld_early(const T* p, bool early) {
  return early ? __ldcg(p) : *p;
}

// One thread per top-k entry (t, h, j); the 16 entries of a (t, h) list sit
// in one half-warp and see each other through shuffles.
//
// This kernel starts once every prep CTA has passed its own wait, so every
// kernel before prep on the stream (the producers of the top-k ids and of
// cu_seqlens) is complete.  With d.early, the inputs -- the entry,
// cu_seqlens and the block_table entry -- are read before this kernel's
// wait, which then covers only prep's outputs (row offsets, status, the
// cleared bitmap).
// Reads before the wait go to L2 (ld.global.cg): the wait is what makes
// earlier kernels' writes visible to plain loads.
__global__ void __launch_bounds__(256) plan_mark_kernel(PlanDev d) {
  if (!d.early) {
    pdl_wait();
    pdl_trigger();
  }
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)d.T * d.Hkv * kTopK;
  const int lane = threadIdx.x & 31;
  const int j = lane & (kTopK - 1);
  const bool live = e < total;
  const int64_t w = e / kTopK;
  const int32_t p = live ? ld_early(d.topk + topk_index(d, w, j), d.early) : -1;
  // prep's plan-valid flag: with the entry when the wait is behind us
  int valid_plan = d.early ? 0 : d.counters[2];
  __shared__ int32_t s_cuq[kMetaCache + 1], s_cuk[kMetaCache + 1], s_off[kMetaCache + 1];
  // (beyond kMetaCache requests, the metadata is read from global memory
  // after the wait); the row offsets are prep's: staged with cu_seqlens
  // when the wait is behind us, after it otherwise
  const bool cache = d.B < kMetaCache;
  if (cache) {
    for (int i = threadIdx.x; i <= d.B; i += blockDim.x) {
      s_cuq[i] = ld_early(d.cu_q + i, d.early);
      s_cuk[i] = ld_early(d.cu_k + i, d.early);
      if (!d.early) s_off[i] = d.req_off[i];
    }
  }
  __syncthreads();
  const ReqMeta m{cache ? s_cuq : d.cu_q, cache ? s_cuk : d.cu_k, cache ? s_off : d.req_off};
  // ids of the same list at positions before j
  bool dup = false;
#pragma unroll
  for (int q = 0; q < kTopK; ++q) {
    const int32_t o = __shfl_sync(0xffffffffu, p, (lane & ~(kTopK - 1)) + q);
    dup |= (q < j) && (o == p);
  }
  const int t = (int)(w / d.Hkv);
  const int h = (int)(w % d.Hkv);
  TokenInfo k = {};
  int32_t phys = -1;
  if (cache && live && d.B > 0) {
    k = token_info_noff(d, m, t);
    // within the row and the table whatever the (not yet checked) seqlens
    if (p >= 0 && p < k.P && p < d.bt_stride && !dup)
      phys = ld_early(d.block_table + (int64_t)k.b * d.bt_stride + p, d.early);
  }
  if (d.early) {
    pdl_wait();
    pdl_trigger();
    valid_plan = d.counters[2];
    if (cache) {
      for (int i = threadIdx.x; i <= d.B; i += blockDim.x) s_off[i] = d.req_off[i];
      __syncthreads();
    }
  }
  if (!cache && live && d.B > 0) {
    k = token_info_noff(d, m, t);
    if (p >= 0 && p < k.P && p < d.bt_stride && !dup)
      phys = d.block_table[(int64_t)k.b * d.bt_stride + p];
  }
  bool keep = false;
  if (live && valid_plan == 1) {
    unsigned st = 0;
    if (p != -1) {
      if (p < -1 || p >= k.P) {
        st |= MSA_STATUS_BAD_PAGE_ID;
      } else if (!dup) {
        if (phys < 0 || (int64_t)phys >= d.num_pages) {
          st |= MSA_STATUS_BAD_BLOCK;
        } else if (p <= k.own) {
          keep = true;
          const int64_t row0 = (int64_t)h * d.total_rows + m.req_off[k.b];
          atomicOr(d.bitmap + (row0 + p) * d.W + (k.i >> 5), 1u << (k.i & 31));
        }
      }
    }
    if (st) atomicOr(d.status, st);
  }
  const uint32_t bal = __ballot_sync(0xffffffffu, keep);
  if (live && j == 0)
    d.slot_mask[w] = (uint16_t)((bal >> (lane & ~(kTopK - 1))) & 0xFFFFu);
}

// The rows of a tile, kPass1Rounds rounds at a time: lane `sub` of a row
// holds the 16-byte vectors [sub * per, (sub + 1) * per) of the row (rows
// are 16-byte aligned, W a multiple of 4), so a row is read, and its word
// prefixes written, as one contiguous span.  The running count in front of
// each word is the lane's own popcounts plus an exclusive scan over the
// row's lanes.  When a lane has one vector per row, a group's vectors are
// all loaded before the first is used.
constexpr int kPass1Rounds = 4;

// Packed (entries, work items) sums: entries in the high word, work items
// in the low word (both below 2^31, so sums of them cannot carry from one
// word into the other).
__device__ __forceinline__ uint64_t pack_cw(int c, int w) {
  return ((uint64_t)(uint32_t)c << 32) | (uint32_t)w;
}

// Inclusive scan over the CTA of one 64-bit value per thread; every thread
// also receives the total.
__device__ __forceinline__ uint64_t block_incl_scan64(uint64_t v, uint64_t* s_warp,
                                                      uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  __syncthreads();  // s_warp may still be read from a previous scan
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  uint64_t before = 0, all = 0;
#pragma unroll
  for (int i = 0; i < kRowThreads / 32; ++i) {
    const uint64_t x = s_warp[i];
    before += i < warp ? x : 0ull;
    all += x;
  }
  *total = all;
  return before + v;
}

// One CTA per tile of d.tile_rows rows (a whole number of rounds, at least
// rows / kMaxRowTiles: at most kMaxRowTiles tiles), worked in segments of at
// most kMaxTileRows rows.  L = 2^d.lane_shift lanes share a row,
// kRowThreads / L rows per round.  Writes each row's length (row_cnt), the
// running count in front of every word (word_pre), the entries and work
// items in front of each row within its tile (row_loc), and the tile's
// totals (tile_state) for the scatter kernel.
__global__ void __launch_bounds__(kRowThreads) plan_rows_kernel(PlanDev d) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_cnt[kMaxTileRows];
  __shared__ uint64_t s_warp[kRowThreads / 32];
  const int tile = blockIdx.x;
  const int L = 1 << d.lane_shift;
  const int sub = threadIdx.x & (L - 1), k = threadIdx.x >> d.lane_shift;
  const int rp = kRowThreads >> d.lane_shift;  // rows per round
  const int nv = d.W >> 2;
  const int per = (nv + L - 1) >> d.lane_shift;
  const int64_t r0 = (int64_t)tile * d.tile_rows;
  const bool ok = d.counters[2] == 1;

  uint64_t carry = 0;  // entries and work items of the segments before
  for (int s0 = 0; s0 < d.tile_rows; s0 += kMaxTileRows) {
    const int seg = min(kMaxTileRows, d.tile_rows - s0);  // a multiple of rp
    const int rounds = seg / rp;
    const int64_t rs = r0 + s0;
    for (int rd0 = 0; rd0 < rounds; rd0 += kPass1Rounds) {
      uint4 v[kPass1Rounds];
#pragma unroll
      for (int u = 0; u < kPass1Rounds; ++u) {
        const int64_t r = rs + (int64_t)(rd0 + u) * rp + k;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (per == 1 && ok && rd0 + u < rounds && r < d.rows && sub < nv)
          v[u] = reinterpret_cast<const uint4*>(d.bitmap + r * d.W)[sub];
      }
#pragma unroll
      for (int u = 0; u < kPass1Rounds; ++u) {
        const int rd = rd0 + u;
        if (rd >= rounds) break;  // the same for the whole CTA
        const int64_t r = rs + (int64_t)rd * rp + k;
        const bool live = ok && r < d.rows;
        const uint4* __restrict__ words = reinterpret_cast<const uint4*>(d.bitmap + r * d.W);
        int own = 0;
        if (per == 1) {
          own = __popc(v[u].x) + __popc(v[u].y) + __popc(v[u].z) + __popc(v[u].w);
        } else if (live) {
          for (int u0 = 0; u0 < per; u0 += 4) {
            uint4 w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int x = sub * per + u0 + i;
              w4[i] = (u0 + i < per && x < nv) ? words[x] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
              own += __popc(w4[i].x) + __popc(w4[i].y) + __popc(w4[i].z) + __popc(w4[i].w);
          }
        }
        int incl = own;
        for (int o = 1; o < L; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, incl, o, L);
          if (sub >= o) incl += n;
        }
        // every lane takes part in the shuffle (a row past the end has 0)
        const int total = __shfl_sync(0xffffffffu, incl, L - 1, L);
        if (sub == 0) s_cnt[rd * rp + k] = total;
        if (live) {
          int4* __restrict__ pre = reinterpret_cast<int4*>(d.word_pre + r * d.W);
          int run = incl - own;
          for (int i = 0; i < per; ++i) {
            const int x = sub * per + i;
            if (x < nv) {
              const uint4 w1 = per == 1 ? v[u] : words[x];
              int4 o;
              o.x = run; run += __popc(w1.x);
              o.y = run; run += __popc(w1.y);
              o.z = run; run += __popc(w1.z);
              o.w = run; run += __popc(w1.w);
              pre[x] = o;
            }
          }
        }
      }
    }
    __syncthreads();  // s_cnt is complete
    // two rows per thread: lengths and offsets within the tile
    const int i0 = 2 * threadIdx.x;
    const int c0 = i0 < seg ? s_cnt[i0] : 0;
    const int c1 = i0 + 1 < seg ? s_cnt[i0 + 1] : 0;
    const uint64_t p0 = pack_cw(c0, (c0 + d.C - 1) / d.C);
    const uint64_t p1 = pack_cw(c1, (c1 + d.C - 1) / d.C);
    uint64_t all;
    // (the scan's barriers also end every read of s_cnt before the next
    // segment writes it)
    uint64_t ex = carry + block_incl_scan64(p0 + p1, s_warp, &all) - (p0 + p1);
    if (i0 < seg && rs + i0 < d.rows) {
      d.row_cnt[rs + i0] = c0;
      reinterpret_cast<int2*>(d.row_loc)[rs + i0] = make_int2((int)(ex >> 32), (int)(uint32_t)ex);
    }
    ex += p0;
    if (i0 + 1 < seg && rs + i0 + 1 < d.rows) {
      d.row_cnt[rs + i0 + 1] = c1;
      reinterpret_cast<int2*>(d.row_loc)[rs + i0 + 1] =
          make_int2((int)(ex >> 32), (int)(uint32_t)ex);
    }
    carry += all;
  }
  if (threadIdx.x == 0) d.tile_state[tile] = carry;
}

// One thread per top-k entry (at least one per 2048 rows): each CTA first
// adds up the row tiles' totals in shared memory (the exclusive scan across
// tiles, at most kMaxRowTiles of them) and writes its share of row_ptr.  A
// kept entry's place in its row is the number of tokens of the row before
// it, read from the word prefix plus a popcount; its CSR slot and work item
// follow from its tile's base and its row's offsets in the tile.  The first
// entry of each chunk of a row also writes the chunk's work item and record
// header.
__global__ void __launch_bounds__(kRowThreads) plan_scatter_kernel(PlanDev d) {
  // This kernel starts once every rows CTA has passed its own wait, so prep
  // and mark are complete.  With d.early, the entry, its slot mask, the
  // plan-valid flag, the request metadata, the block_table entry and the
  // bitmap word are read before this kernel's wait (through L2:
  // ld.global.cg), which then covers only the rows kernel's outputs.
  if (!d.early) {
    pdl_wait();
    pdl_trigger();
  }
  __shared__ uint64_t s_base[kMaxRowTiles];  // entries << 32 | work items before each tile
  __shared__ uint64_t s_warp[kRowThreads / 32];
  __shared__ int32_t s_cuq[kMetaCache + 1], s_cuk[kMetaCache + 1], s_off[kMetaCache + 1];
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = e < (int64_t)d.T * d.Hkv * kTopK;
  const int64_t w = e / kTopK;
  const int j = (int)(e % kTopK);
  const int32_t p = live ? ld_early(d.topk + topk_index(d, w, j), d.early) : -1;
  const uint32_t mask = live ? ld_early(d.slot_mask + w, d.early) : 0u;
  const int valid_plan = ld_early(d.counters + 2, d.early);
  // this thread's rows of row_ptr: r0, r0 + grid threads, ... (rows < 2^31:
  // 32-bit indices); the first one's offset is loaded with the tile totals:
  // together with the entry when the wait is behind us, after it otherwise
  const int r0 = blockIdx.x * blockDim.x + threadIdx.x;
  uint64_t tv = 0;
  int loc0 = 0;
  auto tiles = [&]() {
    tv = (int)threadIdx.x < d.ntiles ? d.tile_state[threadIdx.x] : 0ull;
    loc0 = r0 < (int)d.rows ? d.row_loc[2 * (int64_t)r0] : 0;
  };
  if (!d.early) tiles();
  const bool cache = d.B < kMetaCache;
  if (cache) {
    for (int i = threadIdx.x; i <= d.B; i += blockDim.x) {
      s_cuq[i] = ld_early(d.cu_q + i, d.early);
      s_cuk[i] = ld_early(d.cu_k + i, d.early);
      s_off[i] = ld_early(d.req_off + i, d.early);
    }
  }
  __syncthreads();
  const ReqMeta m = cache ? ReqMeta{s_cuq, s_cuk, s_off} : ReqMeta{d.cu_q, d.cu_k, d.req_off};
  const bool kept = live && valid_plan == 1 && ((mask >> j) & 1u);
  const int t = (int)(w / d.Hkv);
  const int h = (int)(w % d.Hkv);
  TokenInfo k = {};
  int32_t phys = 0;
  int64_t r = 0, wi = 0;
  uint32_t word = 0;
  auto entry = [&](bool cg) {
    k = token_info(d, m, t, h);
    const int32_t* bt = d.block_table + (int64_t)k.b * d.bt_stride + p;  // checked by mark
    r = k.row0 + p;
    wi = r * d.W + (k.i >> 5);
    phys = cg ? __ldcg(bt) : *bt;
    word = cg ? __ldcg(d.bitmap + wi) : d.bitmap[wi];
  };
  if (kept && cache) entry(d.early);
  if (d.early) {
    pdl_wait();
    pdl_trigger();
    tiles();
  }
  if (kept && !cache) entry(false);
  // a kept entry's loads of the rows kernel's outputs go out before the
  // tiles' scan
  int2 loc = make_int2(0, 0);
  int cnt = 0, pre = 0;
  if (kept) {
    loc = reinterpret_cast<const int2*>(d.row_loc)[r];
    cnt = d.row_cnt[r];
    pre = d.word_pre[wi];
  }
  uint64_t all;
  const uint64_t tin = block_incl_scan64(tv, s_warp, &all);
  if ((int)threadIdx.x < d.ntiles) s_base[threadIdx.x] = tin - tv;
  __syncthreads();
  if (r0 < (int)d.rows) d.row_ptr[r0] = (int)(s_base[r0 / d.tile_rows] >> 32) + loc0;
  for (int rr = r0 + gridDim.x * blockDim.x; rr < (int)d.rows; rr += gridDim.x * blockDim.x)
    d.row_ptr[rr] = (int)(s_base[rr / d.tile_rows] >> 32) + d.row_loc[2 * (int64_t)rr];
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // the totals, and the CSR's closing entry
    d.counters[0] = (int)(all >> 32);
    d.counters[1] = (int)(uint32_t)all;
    d.row_ptr[d.rows] = (int)(all >> 32);
  }
  if (!kept) return;
  const uint32_t below = (1u << (k.i & 31)) - 1u;
  const int rank = pre + __popc(word & below);
  const uint64_t base = s_base[(int)r / d.tile_rows];
  const int at = (int)(base >> 32) + loc.x + rank;
  const int64_t rec = (int64_t)(uint32_t)base + loc.y + rank / d.C;
  d.q_idx[at] = t;
  d.slot[at] = (uint8_t)j;
  d.records[rec * d.rec_stride + 1 + rank % d.C] = make_int4(t, k.pos, j, 0);
  if (rank % d.C == 0) {
    const int n = min(d.C, cnt - rank);
    reinterpret_cast<int4*>(d.work)[rec] = make_int4(at, n, k.b, (h << 24) | p);
    // record header: KV tile row of the pool, token count, first key
    // position of the page, first query head of the KV head
    d.records[rec * d.rec_stride] = make_int4((phys * d.Hkv + h) * kPage, n, p * kPage, h * d.G);
  }
}

}  // namespace

cudaError_t launch_plan(const msa_plan_t& pl, const int32_t* topk,
                        const int32_t* block_table, cudaStream_t stream,
                        int topk_hkv, int h_begin) {
  PlanDev d;
  d.topk = topk;
  d.topk_hkv = topk_hkv;
  d.h_begin = h_begin;
  d.cu_q = pl.cu_seqlens_q;
  d.cu_k = pl.cu_seqlens_k;
  d.block_table = block_table;
  d.bt_stride = pl.bt_stride;
  d.num_pages = pl.num_pages;
  d.B = (int)pl.B;
  d.T = (int)pl.T;
  d.Hkv = (int)pl.Hkv;
  d.G = (int)(pl.Hq / pl.Hkv);
  d.W = (int)pl.bitmap_words;
  d.C = (int)pl.chunk_tokens;
  d.total_rows = pl.total_rows;
  d.rows = pl.rows;
  d.max_q = pl.max_seqlen_q;
  d.max_k = pl.max_seqlen_k;
  d.req_off = pl.req_off;
  d.bitmap = pl.bitmap;
  d.word_pre = pl.word_pre;
  d.row_cnt = pl.row_cnt;
  d.row_loc = pl.row_loc;
  d.tile_state = pl.tile_state;
  // Reading inputs before the wait pays when the kernel in front -- prep
  // clearing the bitmap, rows scanning it -- runs long next to that early
  // work, which grows with the top-k entries: measured on GB300, it gains
  // 3 us on plans with 64 and more bitmap bytes per entry (1M-token
  // prefill, decode batches) and loses 1-3 us at 10 and fewer (chunked and
  // ragged prefills); the switch sits at 32.
  d.early = plan_is_sparse(pl.rows, pl.bitmap_words, pl.T, pl.Hkv) ? 1 : 0;
  d.lane_shift = plan_row_lane_shift(pl.bitmap_words);
  d.tile_rows = (int)plan_tile_rows(pl.rows, pl.bitmap_words);
  d.ntiles = (int)ceil_div(pl.rows, d.tile_rows);
  d.row_ptr = pl.row_ptr;
  d.q_idx = pl.q_idx;
  d.slot = pl.slot;
  d.work = pl.work;
  d.records = reinterpret_cast<int4*>(pl.records);
  d.rec_stride = (int)(pl.record_bytes / 16);
  d.counters = pl.counters;
  d.slot_mask = pl.slot_mask;
  d.status = pl.status;

  // bitmap rows are W words, W a multiple of 4: whole 16-byte vectors
  const int64_t bitmap_vec = pl.rows * pl.bitmap_words / 4;
  const int64_t zgrid = std::min<int64_t>(ceil_div(bitmap_vec, kScanThreads),
                                          2 * (int64_t)num_sms());
  const int64_t marks = (int64_t)pl.T * pl.Hkv * kTopK;
  const unsigned mgrid = (unsigned)ceil_div(marks, 256);
  cudaError_t e = launch_pdl(plan_prep_kernel, (unsigned)std::max<int64_t>(zgrid, 1),
                             kScanThreads, 0, stream, d, bitmap_vec);
  if (e == cudaSuccess && marks > 0)
    e = launch_pdl(plan_mark_kernel, mgrid, 256, 0, stream, d);
  if (e == cudaSuccess && d.ntiles > 0)
    e = launch_pdl(plan_rows_kernel, (unsigned)d.ntiles, kRowThreads, 0, stream, d);
  // the scatter kernel also writes row_ptr: at most 2048 rows per CTA
  const unsigned sgrid = (unsigned)std::max<int64_t>(
      std::max<int64_t>(mgrid, ceil_div(pl.rows, 2048)), 1);
  if (e == cudaSuccess)
    e = launch_pdl(plan_scatter_kernel, sgrid, kRowThreads, 0, stream, d);
  return e;
}

}  // namespace msa
