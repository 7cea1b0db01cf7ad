// small_kernels.cu -- the latency-bound kernels of the verify path:
//   subpage_view_kernel   P128 page table -> P32 grouped-HND sub-page indices
//   zero_kernel           zeroes a call's counters inside the launch chain
//   sparse_plan_kernel    per (request, KV head): unique selected blocks, the
//                         bitmask of verify tokens that selected each, and
//                         each block's page slot
//   topk_kernel           warp-level per-token top-k (radix select), ties to
//                         the lower block index, ascending output
//   combine_kernel        split-KV combine: merges the (normalised output,
//                         log2-sum-exp) partials of every sequence that the
//                         attention kernel's stream-K split cut
//   stage_kv_kernel       writes the qo_len verify tokens' K and V into their
//                         cache slots along the ladder
//   flat_table_kernel     flat (CSR) page table <-> padded table, row bases
//                         from the lengths
#include "common.cuh"
#include "launch.h"
#include "plan.cuh"
#include "topk.cuh"

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
  pdl_wait();
  pdl_trigger();
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
// Zeroes n counters once the previous kernel of the stream has finished (a
// kernel, unlike a memset, keeps the launch chain programmatic, so the kernel
// after it is set up while this one runs).
__global__ void zero_kernel(int32_t* __restrict__ c, int n) {
  pdl_trigger();
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) c[i] = 0;
}

cudaError_t launch_zero(int32_t* c, int n, cudaStream_t st) {
  const int threads = 256;
  const int blocks = n / threads + 1 < 64 ? n / threads + 1 : 64;
  return launch_pdl(zero_kernel, dim3(blocks), dim3(threads), 0, st, c, n);
}

// ---------------------------------------------------------------------------
// Sparse plan: one CTA per (request, KV head) sequence builds its plan
// (build_sequence_plan, plan.cuh) from the sequence's T rows of selected
// blocks.
__global__ void sparse_plan_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ lens,
                                   int batch, int qo_len, int num_kv_heads, int max_pages, int topk,
                                   PlanOut out, const int32_t* __restrict__ pt, int num_slots, int* err) {
  extern __shared__ uint32_t mask[];  // [max_pages]
  __shared__ uint32_t bad_tokens;
  __shared__ int32_t warp_tot[32];
  pdl_wait();
  pdl_trigger();
  const int s = blockIdx.x, b = s / num_kv_heads, h = s % num_kv_heads;
  build_sequence_plan(idx, b, h, qo_len, num_kv_heads, topk, max_pages, lens[b], out, pt, num_slots, err, mask,
                      &bad_tokens, warp_tot, threadIdx.x, blockDim.x, [] { __syncthreads(); });
  (void)batch;
}

// ---------------------------------------------------------------------------
// Per-token top-k (the selection itself is topk_row, topk.cuh): one warp per
// (b, t, h) row of n_t = floor((kv_len - qo_len + t) / 128) + 1 valid blocks;
// rows of invalid requests are all -1.
__global__ void topk_kernel(const float* __restrict__ scores, const int32_t* __restrict__ lens,
                            int batch, int qo_len, int num_kv_heads, int max_pages, int topk,
                            int32_t* __restrict__ out, int* err) {
  __shared__ uint32_t hist_all[8][256];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  const int64_t nrows = static_cast<int64_t>(batch) * qo_len * num_kv_heads;
  if (row >= nrows) return;
  const int t = static_cast<int>((row / num_kv_heads) % qo_len);
  const int b = static_cast<int>(row / (static_cast<int64_t>(num_kv_heads) * qo_len));
  const int L = lens[b];
  int n = 0;
  if (len_valid(L, qo_len, max_pages)) n = (L - qo_len + t) / kPage + 1;
  else if (t == 0 && lane == 0 && (row % num_kv_heads) == 0) atomicOr(err, TRTV_DEVERR_KV_LEN);
  topk_row(scores + row * max_pages, n, topk, out + row * topk, hist_all[warp], lane);
}

// ---------------------------------------------------------------------------
// host launchers


// ---------------------------------------------------------------------------
// Split-KV combine.  The attention over a sequence cut into pieces i with
// partial outputs o_i (each normalised by its own softmax sum) and log2-sum-exp
// lse_i equals softmax over the union: o = sum_i 2^(lse_i - M) o_i /
// sum_i 2^(lse_i - M), M = max_i lse_i (the ladder and sparse passes of
// "... verify" attend each row's visible positions exactly once, whichever
// piece holds them).  One CTA per (CTA boundary k, chunk of 32 rows; four
// float4 per thread for head_dim 128, two for 64): boundary k's
// descriptor names the cut sequence it starts (or none); contributors are
// summed in CTA order, so the result does not depend on timing.  Each thread
// holds several elements, so one wave of CTAs covers every cut sequence and
// each thread keeps many independent loads in flight.  Launched with
// programmatic dependent launch right after the attention kernel: the CTAs
// wait (pdl_wait) until that kernel has finished and its partials are visible.
constexpr int kCombineThreads = 256;
// rows per CTA
__host__ __device__ constexpr int combine_rows(int) { return 32; }

template <int D>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __grid_constant__ AttnParams p) {
  constexpr int F4 = D / 4;         // float4 per row
  constexpr int R = combine_rows(D);  // rows of this CTA's chunk
  constexpr int EL = R * F4 / kCombineThreads;  // elements per thread (4 or 2)
  constexpr int CU = 4;             // contributors per batch of loads
  __shared__ int4 desc[2];
  __shared__ int slots[kMaxCombineParts];
  pdl_wait();
  pdl_trigger();
  const int nch = (p.rows_pad + R - 1) / R;
  const int k = 1 + blockIdx.x / nch, chunk = blockIdx.x % nch;
  const int tid = threadIdx.x;
  if (tid < 2) desc[tid] = __ldcg(reinterpret_cast<const int4*>(p.splits + k) + tid);
  __syncthreads();
  // SplitDesc as two int4: {b, h, c_first, nc}, {first_off, pad, W low, W high}
  const int b = desc[0].x, h = desc[0].y, c_first = desc[0].z, nc = desc[0].w;
  if (b < 0) return;
  const int64_t W = static_cast<int64_t>(static_cast<uint32_t>(desc[1].z)) |
                    (static_cast<int64_t>(desc[1].w) << 32);
  const int64_t P = p.num_ctas;
  for (int i = tid; i < nc; i += kCombineThreads) {
    const int64_t c = c_first + i;
    const bool used = W >= P || cta_unit_begin(c, W, P) < cta_unit_begin(c + 1, W, P);
    slots[i] = used ? static_cast<int>(2 * c + (i == 0 ? desc[1].x : 0)) : -1;
  }
  __syncthreads();
  const int rows = p.rows_pad, r0 = chunk * R, s0 = slots[0];  // the first piece always exists
  // one pass per element (row, 4 head dims), online over the contributors:
  // m = running max lse_i, l = sum 2^(lse_i - m), acc = sum 2^(lse_i - m) o_i
  int r[EL], d[EL];
  float m[EL], l[EL];
  float4 acc[EL];
#pragma unroll
  for (int u = 0; u < EL; ++u) {
    const int e = u * kCombineThreads + tid;
    r[u] = r0 + e / F4;
    d[u] = 4 * (e % F4);
    m[u] = -INFINITY;
    l[u] = 0.f;
    acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int i0 = 0; i0 < nc; i0 += CU) {
    float x[EL][CU];
    float4 v[EL][CU];
#pragma unroll
    for (int j = 0; j < CU; ++j) {
      const int sl = i0 + j < nc ? slots[i0 + j] : -1;
      const int64_t sa = sl >= 0 ? sl : s0;
#pragma unroll
      for (int u = 0; u < EL; ++u) {
        const int rr = r[u] < rows ? r[u] : 0;  // rows past the tile (a 16-row tile) read row 0, unused
        x[u][j] = __ldcg(p.ws_lse + sa * rows + rr);
        v[u][j] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + (sa * rows + rr) * D + d[u]));
        if (sl < 0) x[u][j] = -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < EL; ++u) {
      float mn = m[u];
#pragma unroll
      for (int j = 0; j < CU; ++j) mn = fmaxf(mn, x[u][j]);
      if (mn == -INFINITY) continue;
      const float sc = exp2f(m[u] - mn);
      l[u] *= sc;
      acc[u].x *= sc; acc[u].y *= sc; acc[u].z *= sc; acc[u].w *= sc;
#pragma unroll
      for (int j = 0; j < CU; ++j) {
        if (x[u][j] == -INFINITY) continue;
        const float w = exp2f(x[u][j] - mn);
        l[u] += w;
        acc[u].x += w * v[u][j].x; acc[u].y += w * v[u][j].y;
        acc[u].z += w * v[u][j].z; acc[u].w += w * v[u][j].w;
      }
      m[u] = mn;
    }
  }
  const int64_t obase = static_cast<int64_t>(b) * p.qo_len;
#pragma unroll
  for (int u = 0; u < EL; ++u) {
    const int t = r[u] / p.group_pad, gl = r[u] % p.group_pad;
    if (r[u] >= rows || t >= p.qo_len || gl >= p.group) continue;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);  // no visible position in any piece
    if (l[u] > 0.f) {
      const float inv = p.v_scale / l[u];
      a = make_float4(acc[u].x * inv, acc[u].y * inv, acc[u].z * inv, acc[u].w * inv);
    }
    const int64_t orow = ((obase + t) * p.num_q_heads + static_cast<int64_t>(h) * p.group + gl) * D + d[u];
    if (p.out_f32) {
      *reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow) = a;
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + orow) = pk;
    }
  }
}


// ---------------------------------------------------------------------------
// KV slot staging ("Eagle3 for M3 MSA path + CUDA graphs compatibility",
// commit "... verify": KV slot staging generalizes to the causal ladder).
// Verify token t of request b is cache position p = kv_len - qo_len + t; its
// K row for KV head h goes to element ((s stride) 4 + (p % 128) / 32)
// (Hk 32 D) + (h 32 + p % 32) D of the pool, s = page_table[b][p / 128], and
// its V row to the buffer after (s stride + 1).  bf16 caches take the bits;
// FP8 caches take E4M3(x / scale) (binary32 quotient, round to nearest even,
// saturating).  One thread per 16 output bytes.  A request is written only if
// its kv_len is valid and every staged page names a slot of the pool.
template <bool FP8>
__global__ void stage_kv_kernel(const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new,
                                void* __restrict__ pool, const int32_t* __restrict__ pt,
                                const int32_t* __restrict__ lens, int batch, int qo_len, int Hk, int D,
                                int max_pages, int num_slots, int stride, float k_scale, float v_scale,
                                int* err) {
  pdl_wait();
  pdl_trigger();
  constexpr int EPC = FP8 ? 16 : 8;            // elements per 16-byte output chunk
  const int cpr = D / EPC;                     // chunks per (token, head) row
  const int64_t total = static_cast<int64_t>(batch) * qo_len * Hk * 2 * cpr;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(e % cpr);
    int64_t r = e / cpr;
    const int kv = static_cast<int>(r % 2);
    r /= 2;
    const int h = static_cast<int>(r % Hk);
    const int64_t bt = r / Hk;                 // row of k_new / v_new: b * qo_len + t
    const int b = static_cast<int>(bt / qo_len), t = static_cast<int>(bt % qo_len);
    const int L = lens[b];
    if (!len_valid(L, qo_len, max_pages)) {
      if (t == 0 && h == 0 && kv == 0 && c == 0) atomicOr(err, TRTV_DEVERR_KV_LEN);
      continue;
    }
    const int first = (L - qo_len) / kPage, last = (L - 1) / kPage;
    bool ok = true;
    for (int j = first; j <= last; ++j) {
      const int sj = pt[static_cast<int64_t>(b) * max_pages + j];
      ok = ok && sj >= 0 && sj < num_slots;
    }
    if (!ok) {
      if (t == 0 && h == 0 && kv == 0 && c == 0) atomicOr(err, TRTV_DEVERR_PAGE_ID);
      continue;
    }
    const int p = L - qo_len + t;
    const int64_t s = pt[static_cast<int64_t>(b) * max_pages + p / kPage];
    const int64_t buffer = s * stride + kv;
    const int64_t off = ((buffer * kGroups + (p % kPage) / kSub) * Hk + h) * static_cast<int64_t>(kSub) * D +
                        static_cast<int64_t>(p % kSub) * D + static_cast<int64_t>(c) * EPC;
    const __nv_bfloat16* src = (kv ? v_new : k_new) + (bt * Hk + h) * static_cast<int64_t>(D) + c * EPC;
    if constexpr (FP8) {
      const float scale = kv ? v_scale : k_scale;
      const uint4 a = *reinterpret_cast<const uint4*>(src);
      const uint4 bb = *reinterpret_cast<const uint4*>(src + 8);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, bb.x, bb.y, bb.z, bb.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t packed = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t bits = (w[(4 * i + k) / 2] >> (16 * ((4 * i + k) & 1))) & 0xFFFFu;
          const float x = __uint_as_float(bits << 16);
          const __nv_fp8_storage_t code = __nv_cvt_float_to_fp8(x / scale, __NV_SATFINITE, __NV_E4M3);
          packed |= static_cast<uint32_t>(code) << (8 * k);
        }
        o[i] = packed;
      }
      *reinterpret_cast<uint4*>(static_cast<uint8_t*>(pool) + off) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(pool) + off) = *reinterpret_cast<const uint4*>(src);
    }
  }
}

// ---------------------------------------------------------------------------
// Flat (CSR) page table ("Eagle3 for M3 MSA path + CUDA graphs
// compatibility", verify commit, overlap-correction fix: the flat table's row
// layout follows the lengths, so it is rebuilt from the corrected lengths).
// Row b holds n_b = ceil(L_b / 128) pages (0 for L_b <= 0, max_pages past the
// capacity) starting at base_b = sum_{b' < b} n_b'.
//   TO_FLAT:  flat[base_b + j] = pt[b][j] for j < n_b, indptr[b + 1] = base_b + n_b
//   else:     pt[b][j] = flat[base_b + j] for j < n_b, else 0 (slot 0)
// CTA c owns rows [256 c, 256 c + 256): it sums the page counts of all earlier
// rows, scans its own, then copies its rows' entries with coalesced loops.
constexpr int kFlatRows = 256;

__device__ __forceinline__ int flat_pages(int L, int max_pages) {
  if (L <= 0) return 0;
  const int64_t n = (static_cast<int64_t>(L) + kPage - 1) / kPage;
  return n > max_pages ? max_pages : static_cast<int>(n);
}

template <bool TO_FLAT>
__global__ void __launch_bounds__(kFlatRows)
    flat_table_kernel(const int32_t* __restrict__ src, const int32_t* __restrict__ lens, int batch,
                      int qo_len, int max_pages, int32_t* __restrict__ dst, int32_t* __restrict__ indptr,
                      int* err) {
  __shared__ int warp_tot[kFlatRows / 32];
  __shared__ int row_base[kFlatRows], row_n[kFlatRows];
  pdl_wait();
  pdl_trigger();
  const int r0 = blockIdx.x * kFlatRows;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int before = 0;
  for (int b = threadIdx.x; b < r0; b += kFlatRows) before += flat_pages(lens[b], max_pages);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
  if (lane == 0) warp_tot[warp] = before;
  __syncthreads();
  int base = 0;
#pragma unroll
  for (int w = 0; w < kFlatRows / 32; ++w) base += warp_tot[w];
  __syncthreads();
  const int b = r0 + threadIdx.x;
  int n = 0;
  if (b < batch) {
    const int L = lens[b];
    n = flat_pages(L, max_pages);
    if (!len_valid(L, qo_len, max_pages)) atomicOr(err, TRTV_DEVERR_KV_LEN);
  }
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  row_base[threadIdx.x] = base + incl - n;
  row_n[threadIdx.x] = n;
  if (TO_FLAT && indptr != nullptr && b < batch) {
    indptr[b + 1] = base + incl;
    if (b == 0) indptr[0] = 0;
  }
  __syncthreads();
  const int rows = min(kFlatRows, batch - r0);
  const int total = rows * max_pages;
  for (int e = threadIdx.x; e < total; e += kFlatRows) {
    const int r = e / max_pages, j = e % max_pages;
    const int64_t ti = static_cast<int64_t>(r0 + r) * max_pages + j;
    if (TO_FLAT) {
      if (j < row_n[r]) dst[row_base[r] + j] = src[ti];
    } else {
      dst[ti] = j < row_n[r] ? src[row_base[r] + j] : 0;
    }
  }
}

cudaError_t launch_subpage_view(const int32_t* pt, const int32_t* lens, int32_t* k_sub,
                                int32_t* v_sub, int batch, int qo_len, int max_pages,
                                int num_slots, int stride, int* err, cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(batch) * kGroups * max_pages;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 4096 ? (want > 0 ? want : 1) : 4096);
  return launch_pdl(subpage_view_kernel, dim3(blocks), dim3(threads), 0, st, pt, lens, k_sub, v_sub, batch,
                    qo_len, max_pages, num_slots, stride, err);
}

cudaError_t launch_sparse_plan(const int32_t* idx, const int32_t* lens, int batch, int qo_len,
                               int num_kv_heads, int max_pages, int topk, const PlanOut& out,
                               const int32_t* pt, int num_slots, int* err, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(max_pages) * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(sparse_plan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(sparse_plan_kernel, dim3(batch * num_kv_heads), dim3(256), smem, st, idx, lens, batch,
                    qo_len, num_kv_heads, max_pages, topk, out, pt, num_slots, err);
}

cudaError_t launch_topk(const float* scores, const int32_t* lens, int batch, int qo_len,
                        int num_kv_heads, int max_pages, int topk, int32_t* out, int* err,
                        cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(batch) * qo_len * num_kv_heads;
  const int blocks = static_cast<int>((rows + 7) / 8);
  return launch_pdl(topk_kernel, dim3(blocks), dim3(256), 0, st, scores, lens, batch, qo_len, num_kv_heads,
                    max_pages, topk, out, err);
}

cudaError_t launch_combine(int head_dim, const AttnParams& p, cudaStream_t st) {
  if (p.num_ctas < 2) return cudaSuccess;  // no CTA boundary, nothing is cut
  const int nch = (p.rows_pad + combine_rows(head_dim) - 1) / combine_rows(head_dim);
  const dim3 grid(static_cast<unsigned>((p.num_ctas - 1) * nch));
  return head_dim == 64 ? launch_pdl(combine_kernel<64>, grid, dim3(kCombineThreads), 0, st, p)
                        : launch_pdl(combine_kernel<128>, grid, dim3(kCombineThreads), 0, st, p);
}

cudaError_t launch_stage_kv(const void* k_new, const void* v_new, void* pool, const int32_t* pt,
                            const int32_t* lens, int batch, int qo_len, int Hk, int D, int max_pages,
                            int num_slots, int stride, bool fp8, float k_scale, float v_scale, int* err,
                            cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(batch) * qo_len * Hk * 2 * (D / (fp8 ? 16 : 8));
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 4096 ? (want > 0 ? want : 1) : 4096);
  const auto* kn = static_cast<const __nv_bfloat16*>(k_new);
  const auto* vn = static_cast<const __nv_bfloat16*>(v_new);
  return fp8 ? launch_pdl(stage_kv_kernel<true>, dim3(blocks), dim3(threads), 0, st, kn, vn, pool, pt, lens,
                          batch, qo_len, Hk, D, max_pages, num_slots, stride, k_scale, v_scale, err)
             : launch_pdl(stage_kv_kernel<false>, dim3(blocks), dim3(threads), 0, st, kn, vn, pool, pt, lens,
                          batch, qo_len, Hk, D, max_pages, num_slots, stride, k_scale, v_scale, err);
}

cudaError_t launch_flat_table(bool to_flat, const int32_t* src, const int32_t* lens, int batch,
                              int qo_len, int max_pages, int32_t* dst, int32_t* indptr, int* err,
                              cudaStream_t st) {
  const dim3 grid((batch + kFlatRows - 1) / kFlatRows);
  return to_flat ? launch_pdl(flat_table_kernel<true>, grid, dim3(kFlatRows), 0, st, src, lens, batch,
                              qo_len, max_pages, dst, indptr, err)
                 : launch_pdl(flat_table_kernel<false>, grid, dim3(kFlatRows), 0, st, src, lens, batch,
                              qo_len, max_pages, dst, indptr, err);
}

}  // namespace trtv
