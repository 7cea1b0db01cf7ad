// topk.cuh -- warp-level per-token top-k block selection, shared by the top-k
// kernel and the fused proxy + top-k kernel.
//
// Source: "Eagle3 for M3 MSA path + CUDA graphs compatibility" (fork PR #3),
// commit "... verify": top-k gets per-token ladder valid-page counts, so a
// draft token cannot select blocks past its own attend bound.
//
// One warp per (b, t, h) row.  Keys: scores mapped to order-preserving
// uint32 (with -0 folded into +0, so equal scores are equal keys).  A
// 4 x 8-bit radix select finds the k-th largest key tau and how many of the k
// picks must equal tau; a final ballot pass in ascending block order takes
// every key > tau and the lowest-index keys == tau, which writes the output
// already in ascending order.
#pragma once

#include "common.cuh"

namespace trtv {

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Rows of at most this many blocks keep their keys in registers (32 a lane)
// across the passes; longer rows re-read the scores in every pass.
constexpr int kTopkRegPages = 1024;

// The calling warp writes orow[0..topk): the indices of the min(topk, n)
// largest of srow[0..n), ties to the lower index, ascending, padded with -1.
// hist: 256 words of shared memory owned by the warp.  The scores are read
// through L2 (ld.global.cg), so other CTAs of the same kernel may have written
// them (after a fence the caller synchronises on).
static __device__ __noinline__ void topk_row(const float* srow, int n, int topk, int32_t* orow, uint32_t* hist,
                                      int lane) {
  if (n <= topk) {
    for (int i = lane; i < topk; i += 32) orow[i] = i < n ? i : -1;
    return;
  }
  const bool inreg = n <= kTopkRegPages;
  uint32_t kr[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const int i = k * 32 + lane;
    kr[k] = (inreg && i < n) ? order_key(__ldcg(srow + i)) : 0u;
  }
  uint32_t prefix = 0, pmask = 0;
  int remaining = topk;  // picks still to place among keys matching the prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    if (inreg) {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (k * 32 + lane < n && (kr[k] & pmask) == prefix) atomicAdd(&hist[(kr[k] >> shift) & 255u], 1u);
    } else {
      for (int i = lane; i < n; i += 32) {
        const uint32_t key = order_key(__ldcg(srow + i));
        if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
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
  auto take = [&](int i, uint32_t key) {
    const bool eq = i < n && key == prefix;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const int eq_rank = eq_seen + __popc(eqm & ((1u << lane) - 1u));
    const bool sel = i < n && (key > prefix || (eq && eq_rank < remaining));
    const unsigned selm = __ballot_sync(0xffffffffu, sel);
    if (sel) orow[written + __popc(selm & ((1u << lane) - 1u))] = i;
    written += __popc(selm);
    eq_seen += __popc(eqm);
  };
  if (inreg) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (k * 32 < n) take(k * 32 + lane, kr[k]);
  } else {
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      take(i, i < n ? order_key(__ldcg(srow + i)) : 0u);
    }
  }
  for (int i = written + lane; i < topk; i += 32) orow[i] = -1;
}

}  // namespace trtv
