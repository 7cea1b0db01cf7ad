// plan.cuh -- the sparse plan of one (request, KV head) sequence, built by a
// group of threads of one CTA: the plan kernel (a CTA per sequence) and the
// fused proxy-score + top-k kernel (the CTA that completes a sequence's
// selection builds its plan right after).
//
// Source: "Eagle3 for M3 MSA path + CUDA graphs compatibility", verify
// commit (the sparse pass consumes each verify token's selected blocks).
// For sequence (b, h): mask[v] = bitmask of the tokens t whose list selected
// block v; a token whose list holds an index >= max_pages selects nothing
// (its rows are zero) and raises TRTV_DEVERR_BLOCK_IDX; negative entries are
// empty; blocks at or past kv_len are dropped (no token sees them).  Output:
// the ascending unique blocks with their masks and count, and (given the page
// table) each block's slot, a slot outside the pool raising
// TRTV_DEVERR_PAGE_ID and reading as slot 0.  An invalid kv_len gives an empty
// plan (and TRTV_DEVERR_KV_LEN from head 0).
#pragma once

#include "common.cuh"

namespace trtv {

// Threads tid = 0 .. nthr - 1 (whole warps) call it together; `sync` is their
// barrier.  Shared scratch: mask[npages], bad[1], warp_tot[nthr / 32].  `idx`
// rows are [B, T, Hk, topk] and were written before the call (loads bypass
// L1, so a list another warp of the CTA just stored is seen).
template <typename Sync>
__device__ void build_sequence_plan(const int32_t* idx, int b, int h, int T, int Hk, int topk, int max_pages, int L,
                                    const PlanOut& out, const int32_t* pt, int num_slots, int* err, uint32_t* mask,
                                    uint32_t* bad, int32_t* warp_tot, int tid, int nthr, Sync sync) {
  const int s = b * Hk + h;
  if (!len_valid(L, T, max_pages)) {  // L is the same for every thread
    if (tid == 0) {
      out.count[s] = 0;
      if (h == 0) atomicOr(err, TRTV_DEVERR_KV_LEN);
    }
    return;
  }
  const int npages = (L + kPage - 1) / kPage;
  for (int i = tid; i < npages; i += nthr) mask[i] = 0;
  if (tid == 0) *bad = 0;
  sync();
  for (int e = tid; e < T * topk; e += nthr) {
    const int t = e / topk, i = e % topk;
    const int v = __ldcg(idx + ((static_cast<int64_t>(b) * T + t) * Hk + h) * topk + i);
    if (v < 0) continue;
    if (v >= max_pages) {
      atomicOr(bad, 1u << t);
      atomicOr(err, TRTV_DEVERR_BLOCK_IDX);
      continue;
    }
    if (v >= npages) continue;
    atomicOr(&mask[v], 1u << t);
  }
  sync();
  const uint32_t keep_bits = ~*bad;
  // ordered compaction: each thread a contiguous segment
  const int lane = tid & 31, warp = tid >> 5;
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
  sync();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < (nthr + 31) / 32; ++w) {
      const int t = warp_tot[w];
      warp_tot[w] = run;
      run += t;
    }
    out.count[s] = run;
  }
  sync();
  int pos = warp_tot[warp] + incl - local;
  for (int i = lo; i < hi; ++i) {
    const uint32_t m = mask[i] & keep_bits;
    if (m != 0) {
      const int64_t e = static_cast<int64_t>(s) * out.cap + pos;
      out.blocks[e] = i;
      out.masks[e] = m;
      if (out.slots != nullptr) {
        int slot = pt[static_cast<int64_t>(b) * max_pages + i];
        if (slot < 0 || slot >= num_slots) {
          atomicOr(err, TRTV_DEVERR_PAGE_ID);
          slot = 0;
        }
        out.slots[e] = slot;
      }
      ++pos;
    }
  }
  sync();  // the scratch may be reused once every thread is past this point
}

}  // namespace trtv
