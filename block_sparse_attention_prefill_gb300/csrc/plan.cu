// build_k2q_csr on the device: invert the per-token page lists into
// per-(KV head, page) query lists, plus the work list of the attention
// kernel.  (vLLM docs, sparse_attention_msa, MiniMaxM3SparseMSAImpl.forward:
// build_k2q_csr(topk, cu_seqlens_q, cu_seqlens_k, 128, total_rows =
// total_kv_blocks, qhead_per_kv, return_schedule=True); vLLM PR 60930,
// Details / "Host sync": the plan stays on the device, no host copy.)
//
// Steps, all on `stream`, no host synchronisation; every kernel after the
// first is a programmatic dependent launch (its launch overlaps the tail of
// the kernel before it, its work does not):
//   prep     CTA 0: per-request row offsets (sum of page counts), checks,
//            status word; every CTA: clears its share of the (row, token)
//            membership bitmap
//   mark     one thread per top-k entry: validate the id, drop repeats, set
//            one bit per kept page in the membership bitmap; the (token,
//            KV head) list's 16 threads together write its slot mask.  This is the histogram, kept as bits: repeats
//            collapse and the order of arrival cannot change the result.
//   rows     a half-warp per row: row length (popcount of its words) and
//            the running count in front of every word; per 16-row tile, the
//            sums of the lengths and of the chunk counts
//   emit     each CTA adds up the tile sums in front of it; one thread per
//            row: row_ptr and the row's first work item; the work items /
//            record headers of the CTA's rows dealt over all its threads;
//            the last CTA writes the totals
//   scatter  one thread per top-k entry: each kept entry goes to
//            row_ptr + (tokens of the same row before it), found in O(1)
//            from the word prefix and a popcount; it also fills the token
//            slot of the work record the attention kernel will read.
// Every output is a function of the inputs alone: bit-exact and
// deterministic run to run.
#include <algorithm>

#include "common.cuh"

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
  int32_t* word_pre;
  int32_t* row_cnt;
  int32_t* row_wptr;
  int32_t* tile_sums;
  int ntiles;
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
    for (int64_t i = (int64_t)blockIdx.x * kScanThreads + threadIdx.x; i < bitmap_vec;
         i += (int64_t)gridDim.x * kScanThreads)
      bm[i] = make_uint4(0u, 0u, 0u, 0u);
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
    d.row_ptr[d.rows] = 0;  // the fill kernel's last CTA writes the total
  }
}

struct TokenInfo {
  int b, i, pos, own, P;
  int64_t row0;
};

__device__ __forceinline__ TokenInfo token_info(const PlanDev& d, int t, int h) {
  TokenInfo k;
  k.b = upper_index(d.cu_q, d.B, t);
  k.i = t - d.cu_q[k.b];
  const int64_t ql = d.cu_q[k.b + 1] - d.cu_q[k.b];
  const int64_t sl = d.cu_k[k.b + 1] - d.cu_k[k.b];
  k.pos = (int)(sl - ql + k.i);
  k.own = k.pos / kPage;
  k.P = (int)ceil_div(sl, kPage);
  k.row0 = (int64_t)h * d.total_rows + d.req_off[k.b];
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
  // ids of the same list at positions before j
  bool dup = false;
#pragma unroll
  for (int q = 0; q < kTopK; ++q) {
    const int32_t o = __shfl_sync(0xffffffffu, p, (lane & ~(kTopK - 1)) + q);
    dup |= (q < j) && (o == p);
  }
  bool keep = false;
  if (live && d.counters[2] == 1) {
    const int t = (int)(w / d.Hkv);
    const int h = (int)(w % d.Hkv);
    const TokenInfo k = token_info(d, t, h);
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

// kCountTile rows per CTA, a half-warp per row: lane l of the half-warp
// takes the 16-byte vectors [l * per, (l + 1) * per) of the row (rows are
// 16-byte aligned, W a multiple of 4), so the row is read and written as
// one contiguous span.  The running count in front of every word is the
// lane's own popcounts plus an exclusive scan over the 16 lanes.  The CTA's
// sums of the row lengths and chunk counts go to tile_sums.
__global__ void __launch_bounds__(kPlanTile) plan_rows_kernel(PlanDev d) {
  pdl_wait();
  pdl_trigger();
  static_assert(kPlanTile == 16 * kCountTile, "a half-warp per row");
  __shared__ int s_c[kCountTile], s_w[kCountTile];
  const int sub = threadIdx.x & 15, k = threadIdx.x >> 4;
  const int64_t r = (int64_t)blockIdx.x * kCountTile + k;
  const bool live = d.counters[2] == 1 && r < d.rows;
  const int nv = d.W >> 2;
  const int per = (nv + 15) >> 4;
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
  // inclusive scan over the half-warp (all 32 lanes take part)
  int incl = own;
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o, 16);
    if (sub >= o) incl += n;
  }
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
    if (sub == 0) d.row_cnt[r] = total;
  }
  if (sub == 0) {
    s_c[k] = live ? total : 0;
    s_w[k] = live ? (total + d.C - 1) / d.C : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int tc = 0, tw = 0;
#pragma unroll
    for (int i = 0; i < kCountTile; ++i) {
      tc += s_c[i];
      tw += s_w[i];
    }
    d.tile_sums[blockIdx.x] = tc;
    d.tile_sums[d.ntiles + blockIdx.x] = tw;
  }
}

// kPlanTile rows per CTA.  One thread per row finds the row's offsets (the
// sums of the count tiles in front of the CTA plus a block scan)
// and its page; then the CTA's chunks are dealt to all its threads, each
// finding its row by a search over the rows' first chunks, so a row with
// many chunks does not serialise on one thread.
__global__ void __launch_bounds__(kPlanTile) plan_emit_kernel(PlanDev d) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_wex[kPlanTile];     // first chunk of the row, within the CTA
  __shared__ int s_start[kPlanTile];   // first CSR entry of the row
  __shared__ int s_cnt[kPlanTile];
  __shared__ int4 s_hdr[kPlanTile];    // record header without the count
  __shared__ int2 s_item[kPlanTile];   // work item: request, (KV head, page)
  const int64_t r = (int64_t)blockIdx.x * kPlanTile + threadIdx.x;
  const bool ok = d.counters[2] == 1;
  const int c = (ok && r < d.rows) ? d.row_cnt[r] : 0;
  const int chunks = (c + d.C - 1) / d.C;
  int tc, tw;
  const int ex_c = block_excl_scan<kPlanTile>(c, &tc);
  const int ex_w = block_excl_scan<kPlanTile>(chunks, &tw);
  // the rows in front of this CTA: the sums of the count tiles before it,
  // added up by the whole CTA (no separate scan kernel)
  const int tile0 = blockIdx.x * (kPlanTile / kCountTile);
  __shared__ int s_red[2][kPlanTile / 32];
  int pc = 0, pw = 0;
  for (int i = threadIdx.x; i < tile0; i += kPlanTile) {
    pc += d.tile_sums[i];
    pw += d.tile_sums[d.ntiles + i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pc += __shfl_xor_sync(0xffffffffu, pc, o);
    pw += __shfl_xor_sync(0xffffffffu, pw, o);
  }
  if ((threadIdx.x & 31) == 0) {
    s_red[0][threadIdx.x >> 5] = pc;
    s_red[1][threadIdx.x >> 5] = pw;
  }
  __syncthreads();
  int base_c = 0, base_w = 0;
#pragma unroll
  for (int w = 0; w < kPlanTile / 32; ++w) {
    base_c += s_red[0][w];
    base_w += s_red[1][w];
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
    // the last CTA closes the CSR and publishes the totals
    d.counters[0] = base_c + tc;
    d.counters[1] = base_w + tw;
    d.row_ptr[d.rows] = base_c + tc;
  }
  s_wex[threadIdx.x] = ex_w;
  s_start[threadIdx.x] = base_c + ex_c;
  s_cnt[threadIdx.x] = c;
  if (r < d.rows) {
    d.row_ptr[r] = base_c + ex_c;
    d.row_wptr[r] = base_w + ex_w;
    if (c > 0) {
      const int h = (int)(r / d.total_rows);
      const int64_t rr = r - (int64_t)h * d.total_rows;
      const int b = upper_index(d.req_off, d.B, rr);
      const int p = (int)(rr - d.req_off[b]);
      const int32_t phys = d.block_table[(int64_t)b * d.bt_stride + p];
      // record header: KV tile row of the pool, (token count), first key
      // position of the page, first query head of the KV head
      s_hdr[threadIdx.x] = make_int4((phys * d.Hkv + h) * kPage, 0, p * kPage, h * d.G);
      s_item[threadIdx.x] = make_int2(b, (h << 24) | p);
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < tw; k += kPlanTile) {
    const int j = upper_index(s_wex, kPlanTile, k);  // last row starting at or before k
    const int ch = k - s_wex[j];
    const int n = min(d.C, s_cnt[j] - ch * d.C);
    const int64_t wi = (int64_t)base_w + k;
    reinterpret_cast<int4*>(d.work)[wi] =
        make_int4(s_start[j] + ch * d.C, n, s_item[j].x, s_item[j].y);
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
  if (e >= (int64_t)d.T * d.Hkv * kTopK) return;
  if (d.counters[2] != 1) return;
  const int64_t w = e / kTopK;
  const int j = (int)(e % kTopK);
  if (!((d.slot_mask[w] >> j) & 1u)) return;
  const int t = (int)(w / d.Hkv);
  const int h = (int)(w % d.Hkv);
  const TokenInfo k = token_info(d, t, h);
  const int64_t r = k.row0 + d.topk[e];
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
  d.tile_sums = pl.tile_sums;
  d.ntiles = (int)ceil_div(pl.rows, kCountTile);
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
    e = launch_pdl(plan_rows_kernel, (unsigned)d.ntiles, kPlanTile, 0, stream, d);
  const unsigned egrid = (unsigned)ceil_div(pl.rows, kPlanTile);
  if (e == cudaSuccess && egrid > 0)
    e = launch_pdl(plan_emit_kernel, egrid, kPlanTile, 0, stream, d);
  if (e == cudaSuccess && marks > 0)
    e = launch_pdl(plan_scatter_kernel, mgrid, 256, 0, stream, d);
  return e;
}

}  // namespace msa
