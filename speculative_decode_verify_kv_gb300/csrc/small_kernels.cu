// small_kernels.cu -- the latency-bound kernels of the verify path:
//   subpage_view_kernel   P128 page table -> P32 grouped-HND sub-page indices
//   sparse_plan_kernel    per (request, KV head): unique selected blocks and
//                         the bitmask of verify tokens that selected each
//   topk_kernel           warp-level per-token top-k (radix select), ties to
//                         the lower block index, ascending output
#include "common.cuh"
#include "launch.h"

namespace trtv {

// ---------------------------------------------------------------------------
// Sub-page view ("wrap up eagle changes in m3 side branch", view and
// copy_batch_block_offsets commits; "Default Minimax-m3 to unified draft-target
// kv manager", grouped-HND section).  Entry j of request b: slot
// s = page_table[b][j / 4] while j < ceil(kv_len / 32), else 0;
// K = 4 (s stride) + j % 4, V = 4 (s stride + 1) + j % 4.
__global__ void subpage_view_kernel(const int32_t* __restrict__ pt, const int32_t* __restrict__ lens,
                                    int32_t* __restrict__ k_sub, int32_t* __restrict__ v_sub,
                                    int batch, int qo_len, int max_pages, int num_slots, int stride,
                                    int* err) {
  const int nsub = kGroups * max_pages;
  const int64_t total = static_cast<int64_t>(batch) * nsub;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(e / nsub), j = static_cast<int>(e % nsub);
    const int L = lens[b];
    const int64_t used = (static_cast<int64_t>(L) + kSub - 1) / kSub;
    int64_t s = 0;
    if (j < used) {
      s = pt[static_cast<int64_t>(b) * max_pages + j / kGroups];
      if (s < 0 || s >= num_slots) atomicOr(err, TRTV_DEVERR_PAGE_ID);
    }
    if (j == 0 && !len_valid(L, qo_len, max_pages)) atomicOr(err, TRTV_DEVERR_KV_LEN);
    const int gi = j % kGroups;
    k_sub[e] = static_cast<int32_t>(kGroups * (s * stride) + gi);
    v_sub[e] = static_cast<int32_t>(kGroups * (s * stride + 1) + gi);
  }
}

// ---------------------------------------------------------------------------
// Sparse plan ("Eagle3 for M3 MSA path + CUDA graphs compatibility", verify
// commit: the sparse pass consumes per-row selected blocks).  For sequence
// (b, h): mask[v] = bitmask of tokens t whose list selected block v; a token
// whose list holds an index >= max_pages selects nothing (its rows are zero)
// and raises TRTV_DEVERR_BLOCK_IDX; blocks at or past kv_len are dropped
// (no token sees them).  Output: ascending unique blocks with their masks.
__global__ void sparse_plan_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ lens,
                                   int batch, int qo_len, int num_kv_heads, int max_pages, int topk,
                                   int plan_cap, int32_t* __restrict__ plan_blocks,
                                   uint32_t* __restrict__ plan_masks, int32_t* __restrict__ plan_count,
                                   int* err) {
  extern __shared__ uint32_t mask[];  // [max_pages]
  __shared__ uint32_t bad_tokens;
  __shared__ int32_t warp_tot[32];
  const int s = blockIdx.x, b = s / num_kv_heads, h = s % num_kv_heads;
  const int T = qo_len, L = lens[b];
  if (!len_valid(L, T, max_pages)) {
    if (threadIdx.x == 0) {
      plan_count[s] = 0;
      if (h == 0) atomicOr(err, TRTV_DEVERR_KV_LEN);
    }
    return;
  }
  const int npages = (L + kPage - 1) / kPage;
  for (int i = threadIdx.x; i < npages; i += blockDim.x) mask[i] = 0;
  if (threadIdx.x == 0) bad_tokens = 0;
  __syncthreads();
  for (int e = threadIdx.x; e < T * topk; e += blockDim.x) {
    const int t = e / topk, i = e % topk;
    const int v = idx[((static_cast<int64_t>(b) * T + t) * num_kv_heads + h) * topk + i];
    if (v < 0) continue;
    if (v >= max_pages) {
      atomicOr(&bad_tokens, 1u << t);
      atomicOr(err, TRTV_DEVERR_BLOCK_IDX);
      continue;
    }
    if (v >= npages) continue;
    atomicOr(&mask[v], 1u << t);
  }
  __syncthreads();
  const uint32_t keep_bits = ~bad_tokens;
  // ordered compaction: each thread a contiguous segment
  const int nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = (npages + nthr - 1) / nthr;
  const int lo = min(npages, tid * seg), hi = min(npages, lo + seg);
  int local = 0;
  for (int i = lo; i < hi; ++i) local += (mask[i] & keep_bits) != 0;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < (nthr + 31) / 32; ++w) {
      const int t = warp_tot[w];
      warp_tot[w] = run;
      run += t;
    }
    plan_count[s] = run;
  }
  __syncthreads();
  int pos = warp_tot[warp] + incl - local;
  for (int i = lo; i < hi; ++i) {
    const uint32_t m = mask[i] & keep_bits;
    if (m != 0) {
      plan_blocks[static_cast<int64_t>(s) * plan_cap + pos] = i;
      plan_masks[static_cast<int64_t>(s) * plan_cap + pos] = m;
      ++pos;
    }
  }
}

// ---------------------------------------------------------------------------
// Per-token top-k ("Eagle3 for M3 MSA path + CUDA graphs compatibility",
// verify commit: top-k gets per-token ladder valid-page counts).  One warp
// per (b, t, h) row.  Keys: scores mapped to order-preserving uint32 (with
// -0 folded into +0, so equal scores are equal keys).  A 4 x 8-bit radix
// select finds the k-th largest key tau and how many of the k picks must be
// equal to tau; a final ballot pass in ascending block order takes every key
// > tau and the lowest-index keys == tau, which writes the output already in
// ascending order.
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void topk_kernel(const float* __restrict__ scores, const int32_t* __restrict__ lens,
                            int batch, int qo_len, int num_kv_heads, int max_pages, int topk,
                            int32_t* __restrict__ out, int* err) {
  __shared__ uint32_t hist_all[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  const int64_t nrows = static_cast<int64_t>(batch) * qo_len * num_kv_heads;
  if (row >= nrows) return;
  uint32_t* hist = hist_all[warp];
  const int t = static_cast<int>((row / num_kv_heads) % qo_len);
  const int b = static_cast<int>(row / (static_cast<int64_t>(num_kv_heads) * qo_len));
  const int L = lens[b];
  int n = 0;
  if (len_valid(L, qo_len, max_pages)) n = (L - qo_len + t) / kPage + 1;
  else if (t == 0 && lane == 0 && (row % num_kv_heads) == 0) atomicOr(err, TRTV_DEVERR_KV_LEN);
  const float* srow = scores + row * max_pages;
  int32_t* orow = out + row * topk;
  if (n <= topk) {
    for (int i = lane; i < topk; i += 32) orow[i] = i < n ? i : -1;
    return;
  }
  uint32_t prefix = 0, pmask = 0;
  int remaining = topk;  // picks still to place among keys matching the prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      const uint32_t key = order_key(srow[i]);
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncwarp();
    // lane l owns digits 255 - 8l .. 248 - 8l (descending); counts from the top
    uint32_t cnt[8];
    uint32_t local = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      cnt[k] = hist[255 - 8 * lane - k];
      local += cnt[k];
    }
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t above = incl - local;  // keys in higher digits than this lane's
    int digit = -1;
    uint32_t gt = 0;
    if (above < static_cast<uint32_t>(remaining) && incl >= static_cast<uint32_t>(remaining)) {
      uint32_t run = above;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (digit < 0 && run + cnt[k] >= static_cast<uint32_t>(remaining)) {
          digit = 255 - 8 * lane - k;
          gt = run;
        }
        run += cnt[k];
      }
    }
    const unsigned owner = __ballot_sync(0xffffffffu, digit >= 0);
    const int src = __ffs(owner) - 1;
    digit = __shfl_sync(0xffffffffu, digit, src);
    gt = __shfl_sync(0xffffffffu, gt, src);
    prefix |= static_cast<uint32_t>(digit) << shift;
    pmask |= 255u << shift;
    remaining -= static_cast<int>(gt);
    __syncwarp();
  }
  // tau = prefix; take all keys > tau and the first `remaining` keys == tau
  int written = 0, eq_seen = 0;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    uint32_t key = 0;
    if (i < n) key = order_key(srow[i]);
    const bool eq = i < n && key == prefix;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const int eq_rank = eq_seen + __popc(eqm & ((1u << lane) - 1u));
    const bool sel = i < n && (key > prefix || (eq && eq_rank < remaining));
    const unsigned selm = __ballot_sync(0xffffffffu, sel);
    if (sel) orow[written + __popc(selm & ((1u << lane) - 1u))] = i;
    written += __popc(selm);
    eq_seen += __popc(eqm);
  }
  for (int i = written + lane; i < topk; i += 32) orow[i] = -1;
}

// ---------------------------------------------------------------------------
// host launchers

cudaError_t launch_subpage_view(const int32_t* pt, const int32_t* lens, int32_t* k_sub,
                                int32_t* v_sub, int batch, int qo_len, int max_pages,
                                int num_slots, int stride, int* err, cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(batch) * kGroups * max_pages;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 4096 ? (want > 0 ? want : 1) : 4096);
  subpage_view_kernel<<<blocks, threads, 0, st>>>(pt, lens, k_sub, v_sub, batch, qo_len, max_pages,
                                                  num_slots, stride, err);
  return cudaGetLastError();
}

cudaError_t launch_sparse_plan(const int32_t* idx, const int32_t* lens, int batch, int qo_len,
                               int num_kv_heads, int max_pages, int topk, int plan_cap,
                               int32_t* plan_blocks, uint32_t* plan_masks, int32_t* plan_count,
                               int* err, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(max_pages) * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(sparse_plan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  sparse_plan_kernel<<<batch * num_kv_heads, 256, smem, st>>>(
      idx, lens, batch, qo_len, num_kv_heads, max_pages, topk, plan_cap, plan_blocks, plan_masks,
      plan_count, err);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* scores, const int32_t* lens, int batch, int qo_len,
                        int num_kv_heads, int max_pages, int topk, int32_t* out, int* err,
                        cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(batch) * qo_len * num_kv_heads;
  const int blocks = static_cast<int>((rows + 7) / 8);
  topk_kernel<<<blocks, 256, 0, st>>>(scores, lens, batch, qo_len, num_kv_heads, max_pages, topk,
                                      out, err);
  return cudaGetLastError();
}

}  // namespace trtv
