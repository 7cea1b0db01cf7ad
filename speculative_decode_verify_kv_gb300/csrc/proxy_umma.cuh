// proxy_umma.cuh -- MSA proxy (OnlyScore) block scores on the tcgen05 tensor
// cores, for bf16 K, head_dim 128, G = Hq / Hk a power of two <= 16 and
// G * qo_len <= 128 rows.
//
// Source: "Eagle3 for M3 MSA path + CUDA graphs compatibility" (fork PR #3),
// commit "... verify": the proxy pass is natively multi-token with the
// inclusive causal bound offset kv_len - qo_len.  Score of 128-token page j
// for (b, t, KV head h): max over the group's query heads and the positions p
// of page j with p <= kv_len - qo_len + t of sm_scale * (q . k_p); -inf when
// none qualifies.
//
// Per (request, KV head) sequence the (token, group head) rows form the A
// operand Q[128 x 128] (row = t * G + g; rows past qo_len * G are ignored).
// Per page the K sub-pages form B[128 tokens x 128] and one page costs eight
// UMMA 128x128x16 instructions, S = Q K^T landing in one of two TMEM buffers
// (fp32, lane = row, column = token).
//
// Warp roles (320 threads, one CTA per SM, stream-K over all pages):
//   warp 8     TMA: each sequence's Q tile (3-D box [qo_len][G][64] x 2) and
//              each page's K sub-pages into an NST-stage ring laid out as the
//              UMMA's K-major 128B-swizzled operand: [col block][4][32][128 B].
//   warp 9     lane 0 issues the UMMAs; commits release the K stage, publish
//              the S buffer, and free the Q tile after a sequence's last page.
//   warps 0-7  two epilogue warpgroups take alternate pages: tcgen05.ld of
//              their 128 rows x 128 columns, masked row maximum, maximum over
//              each token's G rows (lane shuffles), one score per token.
// Fused top-k (topk_out set): at the end of each sequence it touched, the CTA
// adds its page count to the sequence's counter; the CTA that completes the
// count selects the top-k blocks of the sequence's qo_len rows (topk_row, one
// epilogue warp per row) from the scores every contributor wrote, and (plan
// set) the sequence's sparse plan from those rows.  Requests with no pages get
// rows of -1 (and empty plans) from CTA b % grid.
#pragma once

#include "attn.cuh"
#include "plan.cuh"
#include "topk.cuh"
#include "umma.cuh"

namespace trtv {

constexpr int kUmmaProxyThreads = 320;
constexpr int kUmmaTmemCols = 256;

template <int D>
__global__ void __launch_bounds__(kUmmaProxyThreads, 1)
    proxy_umma_kernel(const __grid_constant__ CUtensorMap kv_map,
                      const __grid_constant__ CUtensorMap q_map,
                      const __grid_constant__ ProxyParams p) {
  static_assert(D == 128, "tcgen05 proxy handles head_dim 128");
  constexpr int STAGE = kGroups * 2 * kBox;  // one page of K for one head: 32 KB
  // one Q tile: rows x 128 bf16 in two 64-column halves, 16 KB for at most
  // 64 rows (the M = 128 UMMA then reads rows 64..127 from whatever follows
  // the tile, into accumulator rows nobody reads), else 32 KB
  const int QBUF = p.qbuf;
  constexpr uint32_t IDESC = umma_idesc_bf16(128, 128);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int NST = p.nstages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);  // [NST] K page landed
  uint64_t* empty = full + NST;    // [NST] UMMAs finished reading the stage
  uint64_t* tfull = empty + NST;   // [2] S buffer written
  uint64_t* tempty = tfull + 2;    // [2] S buffer read out
  uint64_t* qfull = tempty + 2;    // [2] Q tile landed
  uint64_t* qempty = qfull + 2;    // [2] UMMAs finished with the Q tile
  uint64_t* mdone = qempty + 2;    // [1] every UMMA retired
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mdone + 1);
  int* abortf = reinterpret_cast<int*>(tslot + 1);  // the CTA's give-up flag
  const Waits wt{p.err, abortf, p.wait_ns};
  int32_t* scan = reinterpret_cast<int32_t*>(smem + p.off_scan);
  int32_t* warp_tot = scan + p.batch + 1;
  const int Hk = p.num_kv_heads, T = p.qo_len, NP = p.max_pages, G = p.group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int seq_last;

  pdl_wait();  // inputs may come from the previous kernel of the stream
  // -inf for every score no page pass writes (pages past the request's last
  // page; every page of an invalid request)
  {
    const int64_t total = static_cast<int64_t>(p.batch) * T * Hk * NP;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(kUmmaProxyThreads) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * kUmmaProxyThreads) {
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
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
    }
    mbar_init(mdone, 1);
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
  if (p.topk_out != nullptr) {  // rows of requests without pages select nothing
    for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
      if (scan[b + 1] != scan[b]) continue;
      int32_t* o = p.topk_out + static_cast<int64_t>(b) * T * Hk * p.topk;
      for (int e = threadIdx.x; e < T * Hk * p.topk; e += blockDim.x) o[e] = -1;
      if (p.plan.count != nullptr)
        for (int h = threadIdx.x; h < Hk; h += blockDim.x) p.plan.count[b * Hk + h] = 0;
    }
  }
  if (W == 0) return;
  const int64_t u0 = cta_unit_begin(blockIdx.x, W, p.num_ctas);
  const int64_t u1 = cta_unit_begin(blockIdx.x + 1, W, p.num_ctas);
  if (u0 >= u1) return;

  if (warp == 9) {
    tmem_alloc(tslot, kUmmaTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  uint8_t* qbase = smem + p.off_q;
  uint8_t* kbase = smem + p.off_stage;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&kv_map);
      prefetch_tensormap(&q_map);
      const uint64_t pol = policy_evict_first();
      const int sub_rows = Hk * kSub;
      const uint32_t qbytes = static_cast<uint32_t>(2 * 64 * 2 * G * T);
      int it = 0, sq = 0;
      bool alive = true;
      for (SeqCursor cur = cursor_first(scan, p.batch, Hk, false, u0);
           alive && cur.b < p.batch && cur.start < u1; cursor_next(cur, scan, p.batch, Hk, false), ++sq) {
        const int qb = sq & 1;
        if (sq >= 2 && !mbar_wait(&qempty[qb], static_cast<uint32_t>((sq >> 1) - 1) & 1u, wt)) {
          alive = false;
          break;
        }
        mbar_arrive_expect_tx(&qfull[qb], qbytes);
        for (int hb = 0; hb < 2; ++hb)
          asm volatile(
              "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
              " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(qbase + qb * QBUF + hb * (QBUF / 2))),
              "l"(reinterpret_cast<uint64_t>(&q_map)), "r"(hb * 64), "r"(cur.h * G), "r"(cur.b * T),
              "r"(smem_u32(&qfull[qb]))
              : "memory");
        const int64_t j0 = (u0 > cur.start ? u0 : cur.start) - cur.start;
        const int64_t j1 = ((u1 < cur.start + cur.units) ? u1 : cur.start + cur.units) - cur.start;
        for (int64_t j = j0; j < j1; ++j, ++it) {
          const int st = it % NST;
          const uint32_t ph = static_cast<uint32_t>(it / NST) & 1u;
          if (p.withhold >= 0 && it >= p.withhold) { alive = false; break; }  // tests of the give-up path only
          if (it >= NST && !mbar_wait(&empty[st], ph ^ 1u, wt)) { alive = false; break; }
          int slot = p.page_table[static_cast<int64_t>(cur.b) * NP + j];
          if (slot < 0 || slot >= p.num_slots) {
            atomicOr(p.err, TRTV_DEVERR_PAGE_ID);
            slot = 0;
          }
          uint8_t* dst = kbase + st * STAGE;
          mbar_arrive_expect_tx(&full[st], STAGE);
          const int64_t kbuf = static_cast<int64_t>(slot) * p.slot_stride;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb)
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
              const int y = static_cast<int>((kbuf * kGroups + g) * sub_rows + cur.h * kSub);
              tma_load_2d(dst + (hb * kGroups + g) * kBox, &kv_map, &full[st], hb * 64, y, pol);
            }
        }
      }
      // never leave copies in flight
      for (int k = (it > NST ? it - NST : 0); k < it; ++k)
        mbar_drain(&full[k % NST], static_cast<uint32_t>(k / NST) & 1u, wt);
      if (sq >= 1) mbar_drain(&qfull[(sq - 1) & 1], static_cast<uint32_t>((sq - 1) >> 1) & 1u, wt);
    }
  } else if (warp == 9) {
    // ----------------------------------------------------------- UMMA issuer
    if (lane == 0) {
      int it = 0, sq = 0;
      bool alive = true;
      for (SeqCursor cur = cursor_first(scan, p.batch, Hk, false, u0);
           alive && cur.b < p.batch && cur.start < u1; cursor_next(cur, scan, p.batch, Hk, false), ++sq) {
        const int qb = sq & 1;
        if (!mbar_wait(&qfull[qb], static_cast<uint32_t>(sq >> 1) & 1u, wt)) { alive = false; break; }
        const uint32_t a0 = smem_u32(qbase + qb * QBUF);
        const int64_t j0 = (u0 > cur.start ? u0 : cur.start) - cur.start;
        const int64_t j1 = ((u1 < cur.start + cur.units) ? u1 : cur.start + cur.units) - cur.start;
        for (int64_t j = j0; j < j1; ++j, ++it) {
          const int st = it % NST, buf = it & 1;
          const uint32_t ph = static_cast<uint32_t>(it / NST) & 1u;
          if (!mbar_wait(&full[st], ph, wt)) { alive = false; break; }
          if (it >= 2 && !mbar_wait(&tempty[buf], static_cast<uint32_t>((it >> 1) - 1) & 1u, wt)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t b0 = smem_u32(kbase + st * STAGE);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * (QBUF / 2) + (k & 3) * 32;
            umma_bf16(tmem + buf * 128, umma_desc_sw128(a0 + off),
                      umma_desc_sw128(b0 + (k >> 2) * (STAGE / 2) + (k & 3) * 32), IDESC, k > 0);
          }
          umma_commit(&empty[st]);
          umma_commit(&tfull[buf]);
        }
        umma_commit(&qempty[qb]);
      }
      umma_commit(mdone);
      mbar_drain(mdone, 0, wt);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue
    const int wg = warp >> 2, q = warp & 3;
    const int Gp = p.group_pad;
    const int r = 32 * q + lane;
    const int t = r / Gp, gl = r % Gp;
    const bool valid = t < T && gl < G;
    const bool warp_live = 32 * q < T * Gp;
    bool dead = false;
    int it = 0;
    for (SeqCursor cur = cursor_first(scan, p.batch, Hk, false, u0);
         cur.b < p.batch && cur.start < u1; cursor_next(cur, scan, p.batch, Hk, false)) {
      const int L = p.kv_lens[cur.b];
      const int bound = valid ? L - T + t : -1;
      const int64_t j0 = (u0 > cur.start ? u0 : cur.start) - cur.start;
      const int64_t j1 = ((u1 < cur.start + cur.units) ? u1 : cur.start + cur.units) - cur.start;
      for (int64_t j = j0; j < j1; ++j, ++it) {
        const int buf = it & 1;
        if (buf != wg) continue;
        if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(&tfull[buf], static_cast<uint32_t>(it >> 1) & 1u, wt));
        tc_fence_after();
        float m = -INFINITY;
        if (warp_live) {
          const int pos0 = static_cast<int>(j) * kPage;
          const bool masked = pos0 + kPage - 1 > L - T;
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * 128 + c0, v);
            if (masked) {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj)
                if (pos0 + c0 + jj <= bound) m = fmaxf(m, v[jj]);
            } else {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) m = fmaxf(m, v[jj]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        if (!valid) m = -INFINITY;
        for (int off = 1; off < Gp; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (valid && gl == 0)
          p.scores[((static_cast<int64_t>(cur.b) * T + t) * Hk + cur.h) * NP + j] = m * p.score_scale;
      }
      if (p.topk_out != nullptr) {
        // this CTA's scores of the sequence are written: publish, count, and
        // let the CTA that completes the sequence select its rows
        __threadfence();
        named_barrier(1, 256);
        if (threadIdx.x == 0) {
          const int done = static_cast<int>(j1 - j0);
          const int old = atomicAdd(&p.seq_count[cur.b * Hk + cur.h], done);
          seq_last = old + done == cur.units;
        }
        named_barrier(1, 256);
        if (seq_last) {
          __threadfence();
          for (int tt = warp; tt < T; tt += 8) {
            const int64_t row = (static_cast<int64_t>(cur.b) * T + tt) * Hk + cur.h;
            topk_row(p.scores + row * NP, (L - T + tt) / kPage + 1, p.topk, p.topk_out + row * p.topk,
                     reinterpret_cast<uint32_t*>(smem + p.off_red) + warp * 256, lane);
          }
          if (p.plan.count != nullptr) {
            // the sequence's rows are written: its plan, in the histogram scratch
            uint32_t* scratch = reinterpret_cast<uint32_t*>(smem + p.off_red);
            named_barrier(1, 256);
            build_sequence_plan(p.topk_out, cur.b, cur.h, T, Hk, p.topk, NP, L, p.plan, p.page_table, p.num_slots,
                                p.err, scratch, scratch + 2039, reinterpret_cast<int32_t*>(scratch) + 2040,
                                threadIdx.x, 256, [] { named_barrier(1, 256); });
          }
        }
        named_barrier(1, 256);  // seq_last is rewritten for the next sequence
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kUmmaTmemCols);
  }
}

}  // namespace trtv
