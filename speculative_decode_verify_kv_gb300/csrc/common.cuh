// common.cuh -- device primitives shared by the sm_103a kernels of the
// verify-attention library: mbarrier pipeline with time-bounded waits, TMA
// tiled loads, ldmatrix / mma.sync fragments, FP8 conversion, and the launch
// parameter blocks.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/trtv.h"


namespace trtv {

constexpr int kPage = 128;        // tokens per physical page
constexpr int kSub = 32;          // tokens per sub-page (grouped-HND group)
constexpr int kGroups = 4;        // sub-pages per page
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kBox = 4096;        // bytes of one TMA box: 32 rows x 128 B
constexpr int kMaxCombineParts = 1024;  // upper bound on num_ctas
// tcgen05 attention pipeline depth: one Q tile (16 KB for at most 64 rows,
// else 32 KB), K and V pages of 32 KB (three K stages when they fit)
constexpr int kUmmaAttnQTiles = 1;
constexpr int kUmmaAttnKStagesMax = 3;
constexpr int kUmmaAttnVStages = 3;
constexpr int kUmmaAttnFp8Stages = 6;  // most FP8 K and V pages (16 KB each) per ring
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s bound on any barrier wait
// stream-K setup charge per sequence, in units (pages or blocks)
constexpr int kSeqSetup = 3;       // mma.sync attention
constexpr int kUmmaSeqSetup = 2;   // tcgen05 attention, row-major
constexpr int kPmSeqSetup = 6;     // tcgen05 attention, position-major (a sequence
                                   // switch costs about as much as six pages)

// ---- parameter blocks ----------------------------------------------------

// One CTA boundary of the stream-K split: the sequence (request b, KV head h)
// whose units it cuts first, its contributing CTAs c_first .. c_first + nc - 1
// and the workspace slot offset of the first piece; b = -1 when the boundary
// starts no cut.  Written by the attention CTA that starts at the boundary,
// read by the split-combine kernel.
// Where a sparse plan goes (plan.cuh): ascending unique blocks, token masks
// and page slots of every (request, KV head) sequence, and their counts.
struct PlanOut {
  int32_t* blocks;    // [n_seq, cap]
  uint32_t* masks;    // [n_seq, cap]
  int32_t* count;     // [n_seq]
  int32_t* slots;     // [n_seq, cap] or null
  int cap;
};

struct SplitDesc {
  int b, h, c_first, nc, first_off, pad;
  long long W;  // total units of the call
};

struct AttnParams {
  const __nv_bfloat16* q;
  const int32_t* page_table;
  const int32_t* kv_lens;
  void* out;
  float* ws_o;          // [2 * num_ctas, rows_pad, D] partial outputs
  float* ws_lse;        // [2 * num_ctas, rows_pad] partial log2-sum-exp
  SplitDesc* splits;    // [num_ctas] boundary k's cut sequence (entry 0 unused)
  const int32_t* plan_blocks;   // sparse: [n_seq, plan_cap] selected blocks
  const uint32_t* plan_masks;   // sparse: [n_seq, plan_cap] token bitmasks
  const int32_t* plan_count;    // sparse: [n_seq]
  // sparse with a page table: [n_seq, plan_cap] page-table slot of each
  // selected block (checked by the plan kernel), so a page costs one load
  const int32_t* plan_slots;
  int* err;
  int batch, qo_len, num_q_heads, num_kv_heads, group, group_pad, head_dim;
  int max_pages, num_slots, slot_stride, rows, rows_pad;
  int plan_cap, sparse, out_f32, num_ctas, nstages;
  float scale_log2;     // sm_scale * k_scale * log2(e)
  float v_scale;
  // dynamic shared memory carve-up (byte offsets from the 1024-aligned base)
  int off_stage, stage_bytes, off_k, off_v, off_conv, off_merge, off_ml, off_scan, off_bar;
  int off_q, off_vring, nv, nq;  // tcgen05 kernel: Q tiles (nq), V ring (nv); K ring at off_stage, nstages
  int qbuf;                      // tcgen05 kernel: bytes of one Q tile (rows x 256)
  int off_qf8;                   // tcgen05 kernel, FP8 caches: E4M3 Q tile (rows x 128 B)
  // position-major tcgen05 kernel: P^T regions (np buffers of 2 * rows_pad
  // bytes in 128-byte rows) and log2 of the group
  int off_p, np, lg_group;
  int setup;                     // virtual units charged per sequence start (stream-K weight)
  // P32 sub-page tables (drafter attention): when set, group g of logical page
  // j of request b is sub-page sub_k[b][4 j + g] (V: sub_v) of the pool, and
  // page_table is not read.  num_subpages bounds the entries.
  const int32_t* sub_k;
  const int32_t* sub_v;
  int num_subpages;
  // bounded waits: give-up time of every barrier wait, and (tests of that
  // path only, else -1) the number of pages after which the K producer of
  // each CTA withholds its loads, so that its consumers' waits run out
  uint64_t wait_ns;
  int withhold;
};

struct ProxyParams {
  const __nv_bfloat16* q;
  const int32_t* page_table;
  const int32_t* kv_lens;
  float* scores;
  int* err;
  int batch, qo_len, num_q_heads, num_kv_heads, group, group_pad, head_dim;
  int max_pages, num_slots, slot_stride, rows, rows_pad, num_ctas, nstages;
  float score_scale;    // sm_scale * k_scale (> 0, so it commutes with max)
  int off_stage, stage_bytes, off_red, off_scan, off_bar;
  int off_q;            // tcgen05 path: two Q tiles of qbuf bytes (64 or 128 rows x 128 bf16)
  int qbuf;
  // fused top-k (tcgen05 path): when topk_out is set, the CTA that finishes
  // the last page of a (request, KV head) sequence selects its rows' blocks
  // (8 warps x 256 histogram words at off_red); seq_count[b * Hk + h] counts
  // the pages done (zero before the launch)
  int32_t* topk_out;
  int32_t* seq_count;
  int topk;
  // with topk_out: when plan.count is set, that CTA also builds the sequence's
  // sparse plan (plan.cuh) in the histogram scratch (max_pages <= 2032)
  PlanOut plan;
  uint64_t wait_ns;     // as in AttnParams
  int withhold;
};

// ---- small helpers -------------------------------------------------------

// Programmatic dependent launch: let the next kernel of the stream start
// (trigger), and wait until the previous one has finished and its writes are
// visible (wait; a no-op when the kernel was launched without the attribute).
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Entry i of a P32 sub-page table (sub-page i % (4 max_pages) of its
// request, positions from 32 that on), used when that sub-page starts below
// the request's length L; an unused entry is not read and gives sub-page 0,
// a used entry outside [0, limit) flags the error word and gives sub-page 0.
__device__ __forceinline__ int p32_entry(const int32_t* tab, int64_t i, int j, int L, int limit,
                                         int* err) {
  if (j * 32 >= L) return 0;
  int s = tab[i];
  if (s < 0 || s >= limit) {
    atomicOr(err, TRTV_DEVERR_PAGE_ID);
    s = 0;
  }
  return s;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- mbarrier ------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may stay suspended (not issuing) for up
// to kSuspendNs while the phase is incomplete; it resumes when it completes.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Bounded waits of one CTA.  A wait gives up after `limit_ns` (kWaitNs unless
// a test shortens it): it sets TRTV_DEVERR_TIMEOUT and raises the CTA's abort
// flag, after which every other wait of the CTA gives up at once, so each role
// runs out its loops without waiting and all of them meet at the kernel's last
// barrier.  The loops' barrier counts never depend on whether a wait gave up.
// Drains -- a producer waiting for the copies it issued, the UMMA issuer for
// its last instructions -- ignore the flag and keep the full bound: what they
// wait for was issued and always completes.
struct Waits {
  int* err;             // the device error word
  volatile int* abort;  // shared memory, zeroed before the CTA's first wait
  uint64_t limit_ns;
};

// Wait for the phase with the given parity to complete; false when the wait
// gave up (limit reached, or another wait of the CTA gave up before).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Waits& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    // suspended in the wait rather than spinning: the warps that have work
    // keep the issue slots
    if (mbar_try_wait_suspend(bar, parity)) return true;
    if (*w.abort) return false;
    if (global_timer_ns() - t0 > w.limit_ns) {
      atomicOr(w.err, TRTV_DEVERR_TIMEOUT);
      *w.abort = 1;
      return false;
    }
  }
}

// Wait for work this thread issued (copies in flight, committed UMMAs): not
// cut short by the abort flag, bounded by kWaitNs.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, const Waits& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitNs) {
      atomicOr(w.err, TRTV_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// ---- TMA -----------------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- fragments -----------------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool F16>
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// two E4M3 codes (low byte first) -> f16x2 (low half = low byte), exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// bf16 pair -> f16 pair (exact for |x| in the f16 normal range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v);
  float2 f = __bfloat1622float2(b);
  __half2 h = __floats2half2_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&h);
}

// byte offset of 16-byte chunk c of row r inside a 128B-swizzled TMA box
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// ---- work split (shared by the attention and proxy kernels) ----------------

// Units of work of a CTA: [floor(c W / P), floor((c+1) W / P)).
__device__ __forceinline__ int64_t cta_unit_begin(int64_t c, int64_t W, int64_t P) {
  return (c * W) / P;
}

// The CTA whose range holds unit u (largest c with begin(c) <= u).
__device__ __forceinline__ int64_t cta_of_unit(int64_t u, int64_t W, int64_t P) {
  return ((u + 1) * P - 1) / W;
}

// Block-wide exclusive prefix sum of n per-item unit counts into scan[0..n],
// scan[n] = total.  `count(i)` gives item i's units.  All threads of the
// block must call it.
template <typename F>
__device__ void block_exclusive_scan(int n, int32_t* scan, int32_t* warp_tot, F count) {
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int seg = (n + nthr - 1) / nthr;
  const int lo = min(n, tid * seg), hi = min(n, lo + seg);
  int32_t local = 0;
  for (int i = lo; i < hi; ++i) {  // each count is taken once (it may be a global load)
    const int32_t c = count(i);
    scan[i] = c;
    local += c;
  }
  int32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    int32_t run = 0;
    for (int w = 0; w < (nthr + 31) / 32; ++w) {
      int32_t t = warp_tot[w];
      warp_tot[w] = run;
      run += t;
    }
    scan[n] = run;
  }
  __syncthreads();
  int32_t run = warp_tot[warp] + incl - local;
  for (int i = lo; i < hi; ++i) {
    const int32_t c = scan[i];
    scan[i] = run;
    run += c;
  }
  __syncthreads();
}

__device__ __forceinline__ bool len_valid(int L, int T, int max_pages) {
  return L >= T && static_cast<int64_t>(L) <= static_cast<int64_t>(kPage) * max_pages;
}

}  // namespace trtv
