// build_k2q_csr on the device: invert the per-token page lists into
// per-(KV head, page) query lists, plus the work list of the attention
// kernel.  (vLLM docs, sparse_attention_msa, MiniMaxM3SparseMSAImpl.forward:
// build_k2q_csr(topk, cu_seqlens_q, cu_seqlens_k, 128, total_rows =
// total_kv_blocks, qhead_per_kv, return_schedule=True); vLLM PR 60930,
// Details / "Host sync": the plan stays on the device, no host copy.)
//
// Four kernels, all on `stream`, no host synchronisation; every kernel
// after the first is a programmatic dependent launch (its launch overlaps
// the tail of the kernel before it, its work does not):
//   prep     CTA 0: per-request row offsets (sum of page counts), checks,
//            status word, counters; every CTA: clears its share of the
//            (row, token) membership bitmap and of the tile states
//   mark     one thread per top-k entry: validate the id, drop repeats, set
//            one bit per kept page in the membership bitmap; the (token,
//            KV head) list's 16 threads together write its slot mask.  This
//            is the histogram, kept as bits: repeats collapse and the order
//            of arrival cannot change the result.
//   rows     one CTA per tile of rows (at most kMaxRowTiles tiles), tiles
//            taken in launch order from a ticket counter, a half-warp per
//            row: the row's length (popcount of its words) and the running
//            count in front of every word; the tile publishes its totals
//            (entries, work items) and adds up all its predecessors'
//            published totals in parallel (the scan, with no kernel
//            boundary and no chain of waits); then row_ptr, each row's first
//            work item, and the tile's work items and record headers.
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
  uint64_t* tile_state;  // [ntiles] published tile totals (see rows)
  int ntiles, tile_rows;
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
    for (int64_t i = i0; i < d.ntiles; i += stride) d.tile_state[i] = 0ull;
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
    d.counters[3] = 0;      // the rows kernel's tile ticket
    d.row_ptr[d.rows] = 0;  // the rows kernel's last tile writes the total
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

// Tile state word: bit 63 set once published, bits 31..61 the tile's work
// items, bits 0..30 its CSR entries (both below 2^31, checked on the host).
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Exclusive scan of (c, w) over the 16 rows of a round, in warp 0; the
// round's totals come back in *tc / *tw.
__device__ __forceinline__ void scan16(int c, int w, int* exc, int* exw, int* tc,
                                       int* tw) {
  const int lane = threadIdx.x & 31;
  int ic = c, iw = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nc = __shfl_up_sync(0xffffffffu, ic, o);
    const int nw = __shfl_up_sync(0xffffffffu, iw, o);
    if (lane >= o) {
      ic += nc;
      iw += nw;
    }
  }
  *exc = ic - c;
  *exw = iw - w;
  *tc = __shfl_sync(0xffffffffu, ic, 31);
  *tw = __shfl_sync(0xffffffffu, iw, 31);
}

// One CTA per tile of d.tile_rows rows (a multiple of 16, chosen on the
// host so that there are at most kMaxRowTiles tiles while that keeps a tile
// within kMaxRounds rounds), worked in rounds of 16 rows, a half-warp per
// row.
//   pass 1  per round: lane l of the half-warp takes the 16-byte vectors
//           [l * per, (l + 1) * per) of its row (rows are 16-byte aligned,
//           W a multiple of 4), so the row is read and written as one
//           contiguous span; the running count in front of every word is
//           the lane's own popcounts plus an exclusive scan over the 16
//           lanes; the row length and, for a row that has entries, its
//           record header (through block_table) stay in shared memory.
//   totals  the tile publishes its totals (entries, work items) and adds up
//           those of all the tiles before it, read in parallel by the whole
//           CTA: the exclusive scan across tiles, with no kernel boundary and
//           no chain of waits.
//   pass 2  per round, from shared memory only: row_ptr, each row's first
//           work item, and the round's work items and record headers dealt
//           over all threads.
__global__ void __launch_bounds__(kRowThreads) plan_rows_kernel(PlanDev d) {
  pdl_wait();
  pdl_trigger();
  static_assert(kRowThreads == 16 * kRowTile, "a half-warp per row");
  constexpr int kReqCache = 1024;
  __shared__ int s_tile, s_fail;
  __shared__ int s_req[kReqCache + 1];               // req_off, when B fits
  __shared__ int s_cnt[kMaxRounds * kRowTile];
  __shared__ int4 s_hdr[kMaxRounds * kRowTile];      // record header without the count
  __shared__ int2 s_item[kMaxRounds * kRowTile];     // work item: b, (h << 24) | p
  __shared__ int s_exc[kRowTile], s_exw[kRowTile];
  __shared__ int s_red[3][kRowThreads / 32];
  if (threadIdx.x == 0) {
    // tiles in launch order: every predecessor of a tile has started, so
    // waiting for its totals cannot deadlock
    s_tile = atomicAdd(&d.counters[3], 1);
    s_fail = 0;
  }
  const bool cache_req = d.B < kReqCache;
  if (cache_req)
    for (int i = threadIdx.x; i <= d.B; i += kRowThreads) s_req[i] = d.req_off[i];
  __syncthreads();
  const int tile = s_tile;
  const int32_t* req_off = cache_req ? s_req : d.req_off;
  const int sub = threadIdx.x & 15, k = threadIdx.x >> 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool ok = d.counters[2] == 1;
  const int nv = d.W >> 2;
  const int per = (nv + 15) >> 4;
  const int64_t tile_r0 = (int64_t)tile * d.tile_rows;
  const int rounds = d.tile_rows / kRowTile;

  // ---- pass 1: row lengths, word prefixes, record headers
  int tc = 0, tw = 0;  // the tile's totals, kept by lane 0 of each half-warp
  for (int rd = 0; rd < rounds; ++rd) {
    const int64_t r = tile_r0 + rd * kRowTile + k;
    const bool live = ok && r < d.rows;
    const uint4* __restrict__ words = reinterpret_cast<const uint4*>(d.bitmap + r * d.W);
    int own = 0;
    if (live) {
      for (int u0 = 0; u0 < per; u0 += 4) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int x = sub * per + u0 + u;
          v[u] = (u0 + u < per && x < nv) ? words[x] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          own += __popc(v[u].x) + __popc(v[u].y) + __popc(v[u].z) + __popc(v[u].w);
      }
    }
    int incl = own;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o, 16);
      if (sub >= o) incl += n;
    }
    // every lane takes part in the shuffle (a row past the end has 0)
    const int total = __shfl_sync(0xffffffffu, incl, 15, 16);
    if (live) {
      int4* __restrict__ pre = reinterpret_cast<int4*>(d.word_pre + r * d.W);
      int run = incl - own;
      for (int u = 0; u < per; ++u) {
        const int x = sub * per + u;
        if (x < nv) {
          const uint4 v = words[x];
          int4 o;
          o.x = run; run += __popc(v.x);
          o.y = run; run += __popc(v.y);
          o.z = run; run += __popc(v.z);
          o.w = run; run += __popc(v.w);
          pre[x] = o;
        }
      }
    }
    if (sub == 0) {
      const int idx = rd * kRowTile + k;
      s_cnt[idx] = total;
      if (total > 0) {
        tc += total;
        tw += (total + d.C - 1) / d.C;
        const int h = (int)(r / d.total_rows);
        const int64_t rq = r - (int64_t)h * d.total_rows;
        const int b = upper_index(req_off, d.B, rq);
        const int p = (int)(rq - req_off[b]);
        const int32_t phys = d.block_table[(int64_t)b * d.bt_stride + p];
        // record header: KV tile row of the pool, (token count), first key
        // position of the page, first query head of the KV head
        s_hdr[idx] = make_int4((phys * d.Hkv + h) * kPage, 0, p * kPage, h * d.G);
        s_item[idx] = make_int2(b, (h << 24) | p);
      }
    }
  }

  // ---- the tile's totals; publish them; add up the predecessors'
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tc += __shfl_xor_sync(0xffffffffu, tc, o);
    tw += __shfl_xor_sync(0xffffffffu, tw, o);
  }
  if (lane == 0) {
    s_red[0][warp] = tc;
    s_red[1][warp] = tw;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int c = 0, w = 0;
#pragma unroll
    for (int i = 0; i < kRowThreads / 32; ++i) {
      c += s_red[0][i];
      w += s_red[1][i];
    }
    s_red[2][0] = c;
    s_red[2][1] = w;
    st_relaxed_u64(&d.tile_state[tile],
                   (1ull << 63) | ((uint64_t)(uint32_t)w << 31) | (uint32_t)c);
  }
  int pc = 0, pw = 0;
  bool fail = false;
  for (int i = threadIdx.x; i < tile; i += kRowThreads) {
    uint64_t v = ld_relaxed_u64(&d.tile_state[i]);
    if (!(v >> 63)) {
      // bounded wait for a started predecessor to publish (about a second
      // of wall time at most), polling with a back-off: thousands of
      // threads polling L2 flat out would slow the very tiles they wait for
      const uint64_t t0 = global_timer_ns();
      while (!((v = ld_relaxed_u64(&d.tile_state[i])) >> 63)) {
        __nanosleep(200);
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          fail = true;
          break;
        }
      }
    }
    pc += (int)(v & 0x7fffffffu);
    pw += (int)((v >> 31) & 0x7fffffffu);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pc += __shfl_xor_sync(0xffffffffu, pc, o);
    pw += __shfl_xor_sync(0xffffffffu, pw, o);
  }
  __syncthreads();  // s_red[0..1] is reused below
  if (lane == 0) {
    s_red[0][warp] = pc;
    s_red[1][warp] = pw;
  }
  if (fail) s_fail = 1;
  __syncthreads();
  if (s_fail) {
    // a predecessor never published: the plan is incomplete; the attention
    // kernel sees the status bit and does no work
    if (threadIdx.x == 0) atomicOr(d.status, (unsigned)MSA_STATUS_TIMEOUT);
    return;
  }
  int base_c = 0, base_w = 0;
#pragma unroll
  for (int i = 0; i < kRowThreads / 32; ++i) {
    base_c += s_red[0][i];
    base_w += s_red[1][i];
  }
  if (tile == (int)gridDim.x - 1 && threadIdx.x == 0) {
    // the last tile closes the CSR and publishes the totals
    const int all_c = base_c + s_red[2][0], all_w = base_w + s_red[2][1];
    d.counters[0] = all_c;
    d.counters[1] = all_w;
    d.row_ptr[d.rows] = all_c;
  }

  // ---- pass 2: row_ptr, first work items, the work items of each round
  for (int rd = 0; rd < rounds; ++rd) {
    const int64_t r0 = tile_r0 + rd * kRowTile;
    const int* cnt = s_cnt + rd * kRowTile;
    if (warp == 0) {
      const int64_t r = r0 + lane;
      const int c = lane < kRowTile ? cnt[lane] : 0;
      const int ch = (c + d.C - 1) / d.C;
      int exc, exw, rc, rw;
      scan16(c, ch, &exc, &exw, &rc, &rw);
      if (lane < kRowTile) {
        s_exc[lane] = exc;
        s_exw[lane] = exw;
        if (r < d.rows) {
          d.row_ptr[r] = base_c + exc;
          d.row_wptr[r] = base_w + exw;
        }
      }
    }
    __syncthreads();
    const int rw = s_exw[kRowTile - 1] + (cnt[kRowTile - 1] + d.C - 1) / d.C;
    for (int q = threadIdx.x; q < rw; q += kRowThreads) {
      const int j = upper_index(s_exw, kRowTile, q);  // last row starting at or before q
      const int ch = q - s_exw[j];
      const int n = min(d.C, cnt[j] - ch * d.C);
      const int64_t wi = (int64_t)base_w + q;
      const int2 item = s_item[rd * kRowTile + j];
      reinterpret_cast<int4*>(d.work)[wi] =
          make_int4(base_c + s_exc[j] + ch * d.C, n, item.x, item.y);
      int4 hdr = s_hdr[rd * kRowTile + j];
      hdr.y = n;
      d.records[wi * d.rec_stride] = hdr;
    }
    base_c += s_exc[kRowTile - 1] + cnt[kRowTile - 1];
    base_w += rw;
    __syncthreads();  // s_exc / s_exw are rewritten next round
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
  d.tile_rows = (int)plan_tile_rows(pl.rows);
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
  if (e == cudaSuccess && marks > 0)
    e = launch_pdl(plan_scatter_kernel, mgrid, 256, 0, stream, d);
  return e;
}

}  // namespace msa
