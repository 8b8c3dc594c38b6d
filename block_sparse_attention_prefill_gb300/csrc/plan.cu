// build_k2q_csr on the device: invert the per-token page lists into
// per-(KV head, page) query lists, plus the work list of the attention
// kernel.  (vLLM docs, sparse_attention_msa, MiniMaxM3SparseMSAImpl.forward:
// build_k2q_csr(topk, cu_seqlens_q, cu_seqlens_k, 128, total_rows =
// total_kv_blocks, qhead_per_kv, return_schedule=True); vLLM PR 60930,
// Details / "Host sync": the plan stays on the device, no host copy.)
//
// Five kernels, all on `stream`, no host synchronisation; every kernel
// after the first is a programmatic dependent launch (its launch overlaps
// the tail of the kernel before it, its work does not):
//   prep     CTA 0: per-request row offsets (sum of page counts), checks,
//            status word, counters; every CTA: clears its share of the
//            (row, token) membership bitmap
//   mark     one thread per top-k entry: validate the id, drop repeats, set
//            one bit per kept page in the membership bitmap; the (token,
//            KV head) list's 16 threads together write its slot mask.  This
//            is the histogram, kept as bits: repeats collapse and the order
//            of arrival cannot change the result.
//   rows     one CTA per tile of rows (at most kMaxRowTiles tiles while a
//            tile stays within kMaxTileRows rows), 1 to 16 lanes per row by
//            the row's width: the row's length (popcount of its words), the
//            running count in front of every word, and the tile's totals
//            (entries, work items).
//   emit     one CTA per tile: the sum of the totals of the tiles before it
//            (the exclusive scan across tiles: at most kMaxRowTiles loads,
//            all issued at once), a scan over its own rows, then row_ptr,
//            each row's first work item, and the tile's work items and
//            record headers.  A tile waits for no other tile: the kernel
//            boundary orders them.
//   scatter  one thread per top-k entry: each kept entry goes to
//            row_ptr + (tokens of the same row before it), found in O(1)
//            from the word prefix and a popcount; it also fills the token
//            slot of the work record the attention kernel will read.
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
  int64_t total_rows, rows, max_q, max_k;
  int32_t* req_off;
  uint32_t* bitmap;
  int32_t* word_pre;     // [rows * W] tokens of the row before each word
  int32_t* row_cnt;      // [rows] entries of the row
  int32_t* row_wptr;     // [rows] first work item of the row
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
    d.counters[0] = 0;
    d.counters[1] = 0;
    d.counters[2] = st ? 0 : 1;
    d.row_ptr[d.rows] = 0;  // the emit kernel's last tile writes the total
  }
}

struct TokenInfo {
  int b, i, pos, own, P;
  int64_t row0;
};

// Per-request metadata (cu_seqlens_q, cu_seqlens_k, row offsets), copied
// into shared memory by every CTA of the mark and scatter kernels when the
// batch has at most kMetaCache requests, so that a thread's reads of it do
// not add global round trips after its top-k entry; read from global memory
// otherwise.
constexpr int kMetaCache = 512;
struct ReqMeta {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* req_off;
};

__device__ __forceinline__ ReqMeta stage_req_meta(const PlanDev& d, int32_t* s_cuq,
                                                  int32_t* s_cuk, int32_t* s_off) {
  if (d.B >= kMetaCache) return ReqMeta{d.cu_q, d.cu_k, d.req_off};
  for (int i = threadIdx.x; i <= d.B; i += blockDim.x) {
    s_cuq[i] = d.cu_q[i];
    s_cuk[i] = d.cu_k[i];
    s_off[i] = d.req_off[i];
  }
  __syncthreads();
  return ReqMeta{s_cuq, s_cuk, s_off};
}

__device__ __forceinline__ TokenInfo token_info(const PlanDev& d, const ReqMeta& m,
                                                int t, int h) {
  TokenInfo k;
  k.b = upper_index(m.cu_q, d.B, t);
  k.i = t - m.cu_q[k.b];
  const int64_t ql = m.cu_q[k.b + 1] - m.cu_q[k.b];
  const int64_t sl = m.cu_k[k.b + 1] - m.cu_k[k.b];
  k.pos = (int)(sl - ql + k.i);
  k.own = k.pos / kPage;
  k.P = (int)ceil_div(sl, kPage);
  k.row0 = (int64_t)h * d.total_rows + m.req_off[k.b];
  return k;
}

// One thread per top-k entry (t, h, j); the 16 entries of a (t, h) list sit
// in one half-warp and see each other through shuffles.
__global__ void __launch_bounds__(256) plan_mark_kernel(PlanDev d) {
  pdl_wait();
  pdl_trigger();
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)d.T * d.Hkv * kTopK;
  const int lane = threadIdx.x & 31;
  const int j = lane & (kTopK - 1);
  const bool live = e < total;
  const int64_t w = e / kTopK;
  const int32_t p = live ? d.topk[e] : -1;
  const int valid_plan = d.counters[2];
  __shared__ int32_t s_cuq[kMetaCache + 1], s_cuk[kMetaCache + 1], s_off[kMetaCache + 1];
  const ReqMeta m = stage_req_meta(d, s_cuq, s_cuk, s_off);
  // ids of the same list at positions before j
  bool dup = false;
#pragma unroll
  for (int q = 0; q < kTopK; ++q) {
    const int32_t o = __shfl_sync(0xffffffffu, p, (lane & ~(kTopK - 1)) + q);
    dup |= (q < j) && (o == p);
  }
  bool keep = false;
  if (live && valid_plan == 1) {
    const int t = (int)(w / d.Hkv);
    const int h = (int)(w % d.Hkv);
    const TokenInfo k = token_info(d, m, t, h);
    unsigned st = 0;
    if (p != -1) {
      if (p < -1 || p >= k.P) {
        st |= MSA_STATUS_BAD_PAGE_ID;
      } else if (!dup) {
        const int32_t phys = d.block_table[(int64_t)k.b * d.bt_stride + p];
        if (phys < 0 || (int64_t)phys >= d.num_pages) {
          st |= MSA_STATUS_BAD_BLOCK;
        } else if (p <= k.own) {
          keep = true;
          atomicOr(d.bitmap + (k.row0 + p) * d.W + (k.i >> 5),
                   1u << (k.i & 31));
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

// One CTA per tile of d.tile_rows rows (a whole number of rounds; the host
// keeps the tile count within kMaxRowTiles while a tile stays within
// kMaxTileRows rows).  L = 2^d.lane_shift lanes share a row, kRowThreads / L
// rows per round.  Writes each row's length (row_cnt), the running count in
// front of every word (word_pre), and the tile's totals (entries, work
// items) for the emit kernel.
__global__ void __launch_bounds__(kRowThreads) plan_rows_kernel(PlanDev d) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_cnt[kMaxTileRows];
  __shared__ uint64_t s_warp[kRowThreads / 32];
  const int tile = blockIdx.x;
  const int L = 1 << d.lane_shift;
  const int sub = threadIdx.x & (L - 1), k = threadIdx.x >> d.lane_shift;
  const int rp = kRowThreads >> d.lane_shift;  // rows per round
  const int rounds = d.tile_rows / rp;
  const int nv = d.W >> 2;
  const int per = (nv + L - 1) >> d.lane_shift;
  const int64_t r0 = (int64_t)tile * d.tile_rows;
  const bool ok = d.counters[2] == 1;

  for (int rd0 = 0; rd0 < rounds; rd0 += kPass1Rounds) {
    uint4 v[kPass1Rounds];
#pragma unroll
    for (int u = 0; u < kPass1Rounds; ++u) {
      const int64_t r = r0 + (int64_t)(rd0 + u) * rp + k;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (per == 1 && ok && rd0 + u < rounds && r < d.rows && sub < nv)
        v[u] = reinterpret_cast<const uint4*>(d.bitmap + r * d.W)[sub];
    }
#pragma unroll
    for (int u = 0; u < kPass1Rounds; ++u) {
      const int rd = rd0 + u;
      if (rd >= rounds) break;  // the same for the whole CTA
      const int64_t r = r0 + (int64_t)rd * rp + k;
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
  __syncthreads();
  // row lengths out; the tile's totals
  uint64_t mine = 0;
  for (int i = threadIdx.x; i < d.tile_rows; i += kRowThreads) {
    const int c = s_cnt[i];
    if (r0 + i < d.rows) d.row_cnt[r0 + i] = c;
    mine += pack_cw(c, (c + d.C - 1) / d.C);
  }
  uint64_t all;
  block_incl_scan64(mine, s_warp, &all);
  if (threadIdx.x == 0) d.tile_state[tile] = all;
}

// One CTA per tile of the rows kernel, launched after it: adds up the
// totals of the tiles before it (all final by now: the exclusive scan
// across tiles), scans its own rows (two per thread), and writes row_ptr,
// each row's first work item, and the tile's work items and record headers
// dealt over all threads.  The last tile closes the CSR and writes the
// totals.
__global__ void __launch_bounds__(kRowThreads) plan_emit_kernel(PlanDev d) {
  pdl_wait();
  pdl_trigger();
  constexpr int kReqCache = 1024;
  __shared__ int s_req[kReqCache + 1];   // req_off, when B fits
  __shared__ int s_cnt[kMaxTileRows];    // entries of each row
  __shared__ int s_exc[kMaxTileRows];    // first entry in the tile
  __shared__ int s_exw[kMaxTileRows];    // first work item in the tile
  __shared__ int4 s_hdr[kMaxTileRows];   // record header without the count
  __shared__ int2 s_item[kMaxTileRows];  // work item: b, (h << 24) | p
  __shared__ uint64_t s_warp[kRowThreads / 32];
  const int tile = blockIdx.x;
  const int64_t r0 = (int64_t)tile * d.tile_rows;
  const bool cache_req = d.B < kReqCache;
  // the loads that do not depend on one another go out together
  uint64_t pred = 0;
  for (int i = threadIdx.x; i < tile; i += kRowThreads) pred += d.tile_state[i];
  const int i0 = 2 * threadIdx.x;  // this thread's rows: i0, i0 + 1
  int cnt[2];
#pragma unroll
  for (int e = 0; e < 2; ++e)
    cnt[e] = (i0 + e < d.tile_rows && r0 + i0 + e < d.rows) ? d.row_cnt[r0 + i0 + e] : 0;
  if (cache_req)
    for (int i = threadIdx.x; i <= d.B; i += kRowThreads) s_req[i] = d.req_off[i];
  __syncthreads();
  const int32_t* req_off = cache_req ? s_req : d.req_off;
  int32_t phys[2];
  int hb[2], hp[2], hh[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int64_t r = r0 + i0 + e;
    phys[e] = 0;
    hb[e] = hp[e] = hh[e] = 0;
    if (i0 + e < d.tile_rows && r < d.rows) {
      const int h = (int)(r / d.total_rows);
      const int64_t rq = r - (int64_t)h * d.total_rows;
      const int b = upper_index(req_off, d.B, rq);
      const int p = (int)(rq - req_off[b]);
      phys[e] = d.block_table[(int64_t)b * d.bt_stride + p];
      hb[e] = b;
      hp[e] = p;
      hh[e] = h;
    }
  }
  uint64_t base;
  block_incl_scan64(pred, s_warp, &base);
  const int base_c = (int)(base >> 32), base_w = (int)(uint32_t)base;
  const int w0 = (cnt[0] + d.C - 1) / d.C, w1 = (cnt[1] + d.C - 1) / d.C;
  uint64_t all;
  const uint64_t incl = block_incl_scan64(pack_cw(cnt[0] + cnt[1], w0 + w1), s_warp, &all);
  int ex_c = (int)(incl >> 32) - (cnt[0] + cnt[1]);
  int ex_w = (int)(uint32_t)incl - (w0 + w1);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int i = i0 + e;
    const int64_t r = r0 + i;
    if (i < d.tile_rows) {
      s_cnt[i] = cnt[e];
      s_exc[i] = ex_c;
      s_exw[i] = ex_w;
      if (cnt[e] > 0) {
        // record header: KV tile row of the pool, (token count), first key
        // position of the page, first query head of the KV head
        s_hdr[i] = make_int4((phys[e] * d.Hkv + hh[e]) * kPage, 0, hp[e] * kPage,
                             hh[e] * d.G);
        s_item[i] = make_int2(hb[e], (hh[e] << 24) | hp[e]);
      }
      if (r < d.rows) {
        d.row_ptr[r] = base_c + ex_c;
        d.row_wptr[r] = base_w + ex_w;
      }
    }
    ex_c += cnt[e];
    ex_w += e == 0 ? w0 : w1;
  }
  const int tile_w = (int)(uint32_t)all;
  if (tile == (int)gridDim.x - 1 && threadIdx.x == 0) {
    const int all_c = base_c + (int)(all >> 32), all_w = base_w + tile_w;
    d.counters[0] = all_c;
    d.counters[1] = all_w;
    d.row_ptr[d.rows] = all_c;
  }
  __syncthreads();
  for (int q = threadIdx.x; q < tile_w; q += kRowThreads) {
    const int j = upper_index(s_exw, d.tile_rows, q);  // last row starting at or before q
    const int ch = q - s_exw[j];
    const int n = min(d.C, s_cnt[j] - ch * d.C);
    const int64_t wi = (int64_t)base_w + q;
    const int2 item = s_item[j];
    reinterpret_cast<int4*>(d.work)[wi] =
        make_int4(base_c + s_exc[j] + ch * d.C, n, item.x, item.y);
    int4 hdr = s_hdr[j];
    hdr.y = n;
    d.records[wi * d.rec_stride] = hdr;
  }
}

// One thread per kept top-k entry: its place in the row is the number of
// tokens of the row before it, read from the word prefix plus a popcount.
__global__ void __launch_bounds__(256) plan_scatter_kernel(PlanDev d) {
  pdl_wait();
  pdl_trigger();
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = e < (int64_t)d.T * d.Hkv * kTopK;
  const int64_t w = e / kTopK;
  const int j = (int)(e % kTopK);
  // the entry's loads go out together with the metadata's
  const int32_t p = live ? d.topk[e] : -1;
  const uint32_t mask = live ? d.slot_mask[w] : 0u;
  const int valid_plan = d.counters[2];
  __shared__ int32_t s_cuq[kMetaCache + 1], s_cuk[kMetaCache + 1], s_off[kMetaCache + 1];
  const ReqMeta m = stage_req_meta(d, s_cuq, s_cuk, s_off);
  if (!live || valid_plan != 1 || !((mask >> j) & 1u)) return;
  const int t = (int)(w / d.Hkv);
  const int h = (int)(w % d.Hkv);
  const TokenInfo k = token_info(d, m, t, h);
  const int64_t r = k.row0 + p;
  const int64_t wi = r * d.W + (k.i >> 5);
  const uint32_t below = (1u << (k.i & 31)) - 1u;
  const int rank = d.word_pre[wi] + __popc(d.bitmap[wi] & below);
  const int at = d.row_ptr[r] + rank;
  const int64_t rec = d.row_wptr[r] + rank / d.C;
  d.q_idx[at] = t;
  d.slot[at] = (uint8_t)j;
  d.records[rec * d.rec_stride + 1 + rank % d.C] = make_int4(t, k.pos, j, 0);
}

}  // namespace

cudaError_t launch_plan(const msa_plan_t& pl, const int32_t* topk,
                        const int32_t* block_table, cudaStream_t stream) {
  PlanDev d;
  d.topk = topk;
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
  d.row_wptr = pl.row_wptr;
  d.tile_state = pl.tile_state;
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
  plan_prep_kernel<<<(unsigned)std::max<int64_t>(zgrid, 1), kScanThreads, 0, stream>>>(
      d, bitmap_vec);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && marks > 0)
    e = launch_pdl(plan_mark_kernel, mgrid, 256, 0, stream, d);
  if (e == cudaSuccess && d.ntiles > 0)
    e = launch_pdl(plan_rows_kernel, (unsigned)d.ntiles, kRowThreads, 0, stream, d);
  if (e == cudaSuccess && d.ntiles > 0)
    e = launch_pdl(plan_emit_kernel, (unsigned)d.ntiles, kRowThreads, 0, stream, d);
  if (e == cudaSuccess && marks > 0)
    e = launch_pdl(plan_scatter_kernel, mgrid, 256, 0, stream, d);
  return e;
}

}  // namespace msa
