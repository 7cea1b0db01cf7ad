// proxy.cuh -- MSA proxy (OnlyScore) block scores over P128 pages.
//
// Source: "Eagle3 for M3 MSA path + CUDA graphs compatibility" (fork PR #3),
// commit "... verify": the proxy pass runs natively multi-token with the
// inclusive causal bound offset kv_len - qo_len, i.e. token t's bound is
// kv_len - qo_len + t.  Score of 128-token page j for (b, t, KV head h):
//   max over the group's query heads g and positions p of page j with
//   p <= bound of sm_scale * k_scale * (q[b, t, g] . k_p); -inf when no
//   position qualifies.
//
// Same pipeline as the attention kernel but K only: warp 8 streams each
// page's four K sub-pages with TMA; warps 0..7 each own row tile w % MT and
// token slice (w / MT) * 16 MT of every page, compute S = Q K^T with
// mma.sync, reduce the masked maximum over their rows of each verify token,
// and leave it in shared memory.  Before the producer refills a stage it
// reduces the slices' maxima of the page that stage held and writes the
// page's qo_len scores.
#pragma once

#include "common.cuh"
#include "attn.cuh"

namespace trtv {

template <bool FP8, int D, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    proxy_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ ProxyParams p) {
  constexpr bool F16 = FP8;
  constexpr int NB = FP8 ? 1 : (D * 2) / 128;
  constexpr int SUBK = NB * kBox;
  constexpr int TS = 16 * MT;
  constexpr int CH = TS < 32 ? TS : 32;
  constexpr int NCH = TS / CH;
  constexpr int NT = CH / 8;
  constexpr int KS = D / 16;
  constexpr int NSL = kConsumerWarps / MT;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* empty = full + p.nstages;
  int* abortf = reinterpret_cast<int*>(empty + p.nstages);  // the CTA's give-up flag
  const Waits wt{p.err, abortf, p.wait_ns};
  int32_t* scan = reinterpret_cast<int32_t*>(smem + p.off_scan);
  int32_t* warp_tot = scan + p.batch + 1;
  float* red = reinterpret_cast<float*>(smem + p.off_red);  // [NST][8 slices][32 tokens]
  const int Hk = p.num_kv_heads, T = p.qo_len, NST = p.nstages, NP = p.max_pages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();  // inputs may come from the previous kernel of the stream
  // -inf for every score no page pass writes: pages past the request's last
  // page (all pages of an invalid request).
  {
    const int64_t total = static_cast<int64_t>(p.batch) * T * Hk * NP;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * kThreads) {
      const int j = static_cast<int>(e % NP);
      const int b = static_cast<int>(e / (static_cast<int64_t>(NP) * Hk * T));
      const int L = p.kv_lens[b];
      const int npg = len_valid(L, T, NP) ? (L + kPage - 1) / kPage : 0;
      if (j >= npg) p.scores[e] = -INFINITY;
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    *abortf = 0;
    fence_mbar_init();
  }
  block_exclusive_scan(p.batch, scan, warp_tot, [&](int i) -> int32_t {
    const int L = p.kv_lens[i];
    if (len_valid(L, T, NP)) return (L + kPage - 1) / kPage;
    if (blockIdx.x == 0) atomicOr(p.err, TRTV_DEVERR_KV_LEN);
    return 0;
  });
  const int64_t W = static_cast<int64_t>(scan[p.batch]) * Hk;
  pdl_trigger();
  if (W == 0) return;
  const int64_t u0 = cta_unit_begin(blockIdx.x, W, p.num_ctas);
  const int64_t u1 = cta_unit_begin(blockIdx.x + 1, W, p.num_ctas);
  if (u0 >= u1) return;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------- producer + score flush
    __shared__ int st_b[16], st_h[16], st_j[16];
    const uint64_t pol = policy_evict_first();
    if (lane == 0) prefetch_tensormap(&kv_map);
    const int sub_rows = Hk * kSub;
    auto flush = [&](int st) {
      if (lane < T) {
        float v = -INFINITY;
        for (int q = 0; q < NSL; ++q) v = fmaxf(v, red[(st * 8 + q) * 32 + lane]);
        p.scores[((static_cast<int64_t>(st_b[st]) * T + lane) * Hk + st_h[st]) * NP + st_j[st]] = v;
      }
    };
    int it = 0;
    bool alive = true;
    for (SeqCursor cur = cursor_first(scan, p.batch, Hk, false, u0);
         alive && cur.b < p.batch && cur.start < u1; cursor_next(cur, scan, p.batch, Hk, false)) {
      const int64_t j0 = (u0 > cur.start ? u0 : cur.start) - cur.start;
      const int64_t j1 = ((u1 < cur.start + cur.units) ? u1 : cur.start + cur.units) - cur.start;
      for (int64_t j = j0; j < j1; ++j, ++it) {
        const int st = it % NST;
        const uint32_t ph = static_cast<uint32_t>(it / NST) & 1u;
        if (p.withhold >= 0 && it >= p.withhold) { alive = false; break; }  // tests of the give-up path only
        if (it >= NST) {
          const bool ok = mbar_wait(&empty[st], ph ^ 1u, wt);
          if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
          flush(st);
        }
        __syncwarp();
        if (lane == 0) {
          st_b[st] = cur.b;
          st_h[st] = cur.h;
          st_j[st] = static_cast<int>(j);
          int slot = p.page_table[static_cast<int64_t>(cur.b) * NP + j];
          if (slot < 0 || slot >= p.num_slots) {
            atomicOr(p.err, TRTV_DEVERR_PAGE_ID);
            slot = 0;
          }
          uint8_t* dst = smem + p.off_stage + st * p.stage_bytes;
          mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(p.stage_bytes));
          const int64_t kbuf = static_cast<int64_t>(slot) * p.slot_stride;
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            const int y = static_cast<int>((kbuf * kGroups + g) * sub_rows + cur.h * kSub);
#pragma unroll
            for (int hb = 0; hb < NB; ++hb)
              tma_load_2d(dst + (g * NB + hb) * kBox, &kv_map, &full[st], hb * (FP8 ? 128 : 64), y, pol);
          }
        }
        __syncwarp();
      }
    }
    // drain: the last pages' scores
    for (int k = (it > NST ? it - NST : 0); k < it; ++k) {
      const int st = k % NST;
      const bool ok = __all_sync(0xffffffffu,
                                 mbar_wait(&empty[st], static_cast<uint32_t>(k / NST) & 1u, wt));
      if (ok) flush(st);
      else mbar_drain(&full[st], static_cast<uint32_t>(k / NST) & 1u, wt);
    }
    return;
  }

  // ------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  const int mt = warp % MT, sl = warp / MT;
  const int tok0 = sl * TS;
  const int Gp = p.group_pad;
  bool dead = false;
  int it = 0;
  for (SeqCursor cur = cursor_first(scan, p.batch, Hk, false, u0);
       cur.b < p.batch && cur.start < u1; cursor_next(cur, scan, p.batch, Hk, false)) {
    const int b = cur.b, h = cur.h;
    const int64_t j0 = (u0 > cur.start ? u0 : cur.start) - cur.start;
    const int64_t j1 = ((u1 < cur.start + cur.units) ? u1 : cur.start + cur.units) - cur.start;
    const int L = p.kv_lens[b];
    uint32_t qa[KS][4];
    load_q_frags<FP8, D>(p.q, T, p.num_q_heads, p.group, Gp, b, h, mt, qa);
    int bound[2], trow[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int r = mt * 16 + g + 8 * hh;
      const int t = r / Gp, gl = r % Gp;
      const bool ok = t < T && gl < p.group;
      trow[hh] = t;
      bound[hh] = ok ? L - T + t : -1;
    }
    for (int64_t j = j0; j < j1; ++j, ++it) {
      const int st = it % NST;
      const uint32_t ph = static_cast<uint32_t>(it / NST) & 1u;
      if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(&full[st], ph, wt));
      const int pos0 = static_cast<int>(j) * kPage;
      const uint8_t* kst = smem + p.off_stage + st * p.stage_bytes;
      float rmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int ct = tok0 + cc * CH;
        const int sp = ct / kSub, r0 = ct % kSub;
        float s[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
        if constexpr (FP8) {
          const uint8_t* kb = kst + sp * kBox;
#pragma unroll
          for (int jt = 0; jt < NT; ++jt) {
            const int r = r0 + 8 * jt + g;
            const uint4 w0 = *reinterpret_cast<const uint4*>(kb + sw128(r, 2 * c));
            const uint4 w1 = *reinterpret_cast<const uint4*>(kb + sw128(r, 2 * c + 1));
            const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
              mma16816<F16>(s[jt], qa[ks], e4m3x2_to_f16x2(static_cast<uint16_t>(w[ks] & 0xffffu)),
                            e4m3x2_to_f16x2(static_cast<uint16_t>(w[ks] >> 16)));
          }
        } else {
          const uint8_t* kb = kst + sp * SUBK;
          const int mat = lane >> 3, rr = lane & 7;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const int dch = 2 * ks + (mat & 1);
#pragma unroll
            for (int jp = 0; jp < NT / 2; ++jp) {
              const int r = r0 + 8 * (2 * jp + (mat >> 1)) + rr;
              uint32_t b0, b1, b2, b3;
              ldsm_x4(smem_u32(kb + (dch >> 3) * kBox + sw128(r, dch & 7)), b0, b1, b2, b3);
              mma16816<F16>(s[2 * jp], qa[ks], b0, b1);
              mma16816<F16>(s[2 * jp + 1], qa[ks], b2, b3);
            }
          }
        }
#pragma unroll
        for (int jt = 0; jt < NT; ++jt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pos = pos0 + ct + 8 * jt + 2 * c + (e & 1);
            if (pos <= bound[e >> 1]) rmax[e >> 1] = fmaxf(rmax[e >> 1], s[jt][e]);
          }
      }
      // rows -> verify tokens: quad (columns), then the rows of one token
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        rmax[hh] = fmaxf(rmax[hh], __shfl_xor_sync(0xffffffffu, rmax[hh], 1));
        rmax[hh] = fmaxf(rmax[hh], __shfl_xor_sync(0xffffffffu, rmax[hh], 2));
      }
      if (Gp == 16) rmax[0] = rmax[1] = fmaxf(rmax[0], rmax[1]);
      const int span = Gp < 8 ? Gp : 8;  // rows of one token among g = 0..7
      for (int off = 4; off < 4 * span; off <<= 1) {
        rmax[0] = fmaxf(rmax[0], __shfl_xor_sync(0xffffffffu, rmax[0], off));
        rmax[1] = fmaxf(rmax[1], __shfl_xor_sync(0xffffffffu, rmax[1], off));
      }
      float* rd = red + (st * 8 + sl) * 32;
      if (c == 0 && (g % span) == 0) {
        const float sc = p.score_scale;
        if (trow[0] < T) rd[trow[0]] = rmax[0] * sc;
        if (Gp < 16 && trow[1] < T) rd[trow[1]] = rmax[1] * sc;
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
}

}  // namespace trtv
