// build_k2q_csr on the device: invert the per-token page lists into
// per-(KV head, page) query lists, plus the work list of the attention
// kernel.  (vLLM docs, sparse_attention_msa, MiniMaxM3SparseMSAImpl.forward:
// build_k2q_csr(topk, cu_seqlens_q, cu_seqlens_k, 128, total_rows =
// total_kv_blocks, qhead_per_kv, return_schedule=True); vLLM PR 60930,
// Details / "Host sync": the plan stays on the device, no host copy.)
//
// Steps, all on `stream`, no host synchronisation:
//   memset  status word and the membership bitmap
//   prep    per-request row offsets (sum of page counts), input checks
//   mark    one thread per (token, KV head): validate its 16 ids, set one bit
//           per kept page in the (row, token) membership bitmap, write the
//           token's slot mask -- the histogram, kept as bits so that repeats
//           collapse and the order of arrival cannot matter
//   count   popcount of every row (row length) and of every tile of rows
//   scan    exclusive scan of the tile sums (one CTA)
//   fill    per tile: exclusive scan of its rows -> row_ptr; then one warp per
//           row walks the row's bitmap words in order and scatters the token
//           ids (ascending by construction) with their slot j, and writes the
//           row's work items.
// Every output is a function of the inputs alone: bit-exact and
// deterministic run to run.
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
  int B, T, Hkv, W, C;
  int64_t total_rows, rows, max_q, max_k;
  int32_t* req_off;
  uint32_t* bitmap;
  int32_t* row_cnt;
  int32_t* tile_sums;
  int ntiles;
  int32_t* row_ptr;
  int32_t* q_idx;
  uint8_t* slot;
  int32_t* work;
  int32_t* counters;
  uint16_t* slot_mask;
  uint32_t* status;
};

// counters[2] == 1 when the per-request metadata passed the checks.
__global__ void __launch_bounds__(kScanThreads)
plan_prep_kernel(PlanDev d) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  bool overflow = false;
  bool bad = false;
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
    if (st) atomicOr(d.status, st);
    d.counters[0] = 0;
    d.counters[1] = 0;
    d.counters[2] = st ? 0 : 1;
  }
}

__global__ void __launch_bounds__(256) plan_mark_kernel(PlanDev d) {
  const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= (int64_t)d.T * d.Hkv) return;
  const int t = (int)(w / d.Hkv);
  const int h = (int)(w % d.Hkv);
  uint16_t mask = 0;
  if (d.counters[2] == 1) {
    const int b = upper_index(d.cu_q, d.B, t);
    const int i = t - d.cu_q[b];
    const int64_t ql = d.cu_q[b + 1] - d.cu_q[b];
    const int64_t sl = d.cu_k[b + 1] - d.cu_k[b];
    const int64_t pos = sl - ql + i;
    const int own = (int)(pos / kPage);
    const int P = (int)ceil_div(sl, kPage);
    const int64_t row0 = (int64_t)h * d.total_rows + d.req_off[b];
    const int32_t* ids = d.topk + w * kTopK;
    const int32_t* bt = d.block_table + (int64_t)b * d.bt_stride;
    int32_t seen[kTopK];
    unsigned st = 0;
#pragma unroll
    for (int j = 0; j < kTopK; ++j) {
      const int32_t p = ids[j];
      seen[j] = p;
      if (p == -1) continue;
      if (p < -1 || p >= P) { st |= MSA_STATUS_BAD_PAGE_ID; continue; }
      bool dup = false;
#pragma unroll
      for (int k = 0; k < j; ++k) dup |= (seen[k] == p);
      if (dup) continue;
      const int32_t phys = bt[p];
      if (phys < 0 || (int64_t)phys >= d.num_pages) {
        st |= MSA_STATUS_BAD_BLOCK;
        continue;
      }
      if (p > own) continue;
      mask |= (uint16_t)(1u << j);
      atomicOr(d.bitmap + (row0 + p) * d.W + (i >> 5), 1u << (i & 31));
    }
    if (st) atomicOr(d.status, st);
  }
  d.slot_mask[w] = mask;
}

// One CTA per tile of kPlanTile rows; warp k handles rows k*32 .. k*32+31.
__global__ void __launch_bounds__(kPlanTile) plan_count_kernel(PlanDev d) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t tile0 = (int64_t)blockIdx.x * kPlanTile;
  const bool ok = d.counters[2] == 1;
  __shared__ int s_cnt[kPlanTile];
  for (int k = 0; k < 32; ++k) {
    const int local = warp * 32 + k;
    const int64_t r = tile0 + local;
    int c = 0;
    if (ok && r < d.rows) {
      const uint32_t* words = d.bitmap + r * d.W;
      for (int x = lane; x < d.W; x += 32) c += __popc(words[x]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      if (lane == 0) d.row_cnt[r] = c;
    }
    if (lane == 0) s_cnt[local] = (r < d.rows) ? c : 0;
  }
  __syncthreads();
  const int c = s_cnt[threadIdx.x];
  const int chunks = (c + d.C - 1) / d.C;
  int tc, tw;
  block_excl_scan<kPlanTile>(c, &tc);
  block_excl_scan<kPlanTile>(chunks, &tw);
  if (threadIdx.x == 0) {
    d.tile_sums[blockIdx.x] = tc;
    d.tile_sums[d.ntiles + blockIdx.x] = tw;
  }
}

__global__ void __launch_bounds__(kScanThreads) plan_scan_kernel(PlanDev d) {
  for (int which = 0; which < 2; ++which) {
    int32_t* a = d.tile_sums + (int64_t)which * d.ntiles;
    int carry = 0;
    for (int base = 0; base < d.ntiles; base += kScanThreads) {
      const int i = base + threadIdx.x;
      const int v = i < d.ntiles ? a[i] : 0;
      int total;
      const int ex = block_excl_scan<kScanThreads>(v, &total);
      if (i < d.ntiles) a[i] = carry + ex;
      carry += total;
    }
    if (threadIdx.x == 0) {
      d.counters[which] = carry;
      if (which == 0) d.row_ptr[d.rows] = carry;
    }
  }
}

__global__ void __launch_bounds__(kPlanTile) plan_fill_kernel(PlanDev d) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t tile0 = (int64_t)blockIdx.x * kPlanTile;
  const int64_t r_me = tile0 + threadIdx.x;
  const bool ok = d.counters[2] == 1;
  __shared__ int s_start[kPlanTile];
  __shared__ int s_wstart[kPlanTile];
  __shared__ int s_cnt[kPlanTile];
  const int c = (ok && r_me < d.rows) ? d.row_cnt[r_me] : 0;
  const int chunks = (c + d.C - 1) / d.C;
  int tc, tw;
  const int ex_c = block_excl_scan<kPlanTile>(c, &tc);
  const int ex_w = block_excl_scan<kPlanTile>(chunks, &tw);
  const int start = d.tile_sums[blockIdx.x] + ex_c;
  const int wstart = d.tile_sums[d.ntiles + blockIdx.x] + ex_w;
  if (r_me < d.rows) d.row_ptr[r_me] = start;
  s_start[threadIdx.x] = start;
  s_wstart[threadIdx.x] = wstart;
  s_cnt[threadIdx.x] = c;
  __syncthreads();
  if (!ok) return;

  for (int k = 0; k < 32; ++k) {
    const int local = warp * 32 + k;
    const int64_t r = tile0 + local;
    const int cnt = s_cnt[local];
    if (r >= d.rows || cnt == 0) continue;
    const int h = (int)(r / d.total_rows);
    const int64_t rr = r - (int64_t)h * d.total_rows;
    const int b = upper_index(d.req_off, d.B, rr);
    const int p = (int)(rr - d.req_off[b]);
    const int t0 = d.cu_q[b];
    const int pos0 = s_start[local];
    const uint32_t* words = d.bitmap + r * d.W;
    // tokens, in ascending order
    int done = 0;
    for (int base = 0; base < d.W && done < cnt; base += 32) {
      const uint32_t word = (base + lane < d.W) ? words[base + lane] : 0u;
      const int n = __popc(word);
      const int incl = warp_incl_scan(n);
      int at = pos0 + done + incl - n;
      uint32_t bits = word;
      while (bits) {
        const int bit = __ffs(bits) - 1;
        bits &= bits - 1;
        const int t = t0 + (base + lane) * 32 + bit;
        const int32_t* ids = d.topk + ((int64_t)t * d.Hkv + h) * kTopK;
        int j = 0;
        while (j < kTopK - 1 && ids[j] != p) ++j;
        d.q_idx[at] = t;
        d.slot[at] = (uint8_t)j;
        ++at;
      }
      done += __shfl_sync(0xffffffffu, incl, 31);
    }
    // work items of this row
    const int nch = (cnt + d.C - 1) / d.C;
    for (int ch = lane; ch < nch; ch += 32) {
      int4 item;
      item.x = pos0 + ch * d.C;
      item.y = min(d.C, cnt - ch * d.C);
      item.z = b;
      item.w = (h << 24) | p;
      reinterpret_cast<int4*>(d.work)[s_wstart[local] + ch] = item;
    }
  }
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
  d.W = (int)pl.bitmap_words;
  d.C = (int)pl.chunk_tokens;
  d.total_rows = pl.total_rows;
  d.rows = pl.rows;
  d.max_q = pl.max_seqlen_q;
  d.max_k = pl.max_seqlen_k;
  d.req_off = pl.req_off;
  d.bitmap = pl.bitmap;
  d.row_cnt = pl.row_cnt;
  d.tile_sums = pl.tile_sums;
  d.ntiles = (int)ceil_div(pl.rows, kPlanTile);
  d.row_ptr = pl.row_ptr;
  d.q_idx = pl.q_idx;
  d.slot = pl.slot;
  d.work = pl.work;
  d.counters = pl.counters;
  d.slot_mask = pl.slot_mask;
  d.status = pl.status;

  cudaError_t e = cudaMemsetAsync(pl.status, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  const size_t bm = (size_t)pl.rows * (size_t)pl.bitmap_words * sizeof(uint32_t);
  if (bm) {
    e = cudaMemsetAsync(pl.bitmap, 0, bm, stream);
    if (e != cudaSuccess) return e;
  }
  plan_prep_kernel<<<1, kScanThreads, 0, stream>>>(d);
  const int64_t marks = (int64_t)pl.T * pl.Hkv;
  if (marks > 0)
    plan_mark_kernel<<<(unsigned)ceil_div(marks, 256), 256, 0, stream>>>(d);
  if (d.ntiles > 0)
    plan_count_kernel<<<d.ntiles, kPlanTile, 0, stream>>>(d);
  plan_scan_kernel<<<1, kScanThreads, 0, stream>>>(d);
  if (d.ntiles > 0)
    plan_fill_kernel<<<d.ntiles, kPlanTile, 0, stream>>>(d);
  return cudaGetLastError();
}

}  // namespace msa
