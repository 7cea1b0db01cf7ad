// attn_umma.cuh -- ladder verify attention (dense and MSA sparse) on the
// tcgen05 tensor cores, for bf16 K/V, head_dim 128, G = Hq / Hk a power of
// two and G * qo_len <= 128 rows.
//
// Sources: "Eagle3 for M3 MSA path + CUDA graphs compatibility" (fork PR #3),
// commit "... verify" (token t attends kv_len - qo_len + t + 1 positions; the
// sparse pass attends the selected blocks); "Default Minimax-m3 to unified
// draft-target kv manager" (#17835), "Grouped-HND draft KV transfer" (page
// layout); "wrap up eagle changes in m3 side branch" (#18066), view commit
// (K page at slot * stride, V page at slot * stride + 1).
//
// Work split as in attn_kernel (stream-K over the pages / selected blocks of
// every (request, KV head) sequence; cut sequences are merged by the
// split-combine kernel).  Per sequence the (token, group head) rows (row =
// t * G + g) are the UMMA's M -- M = 128, or for tiles of at most 64 bf16 rows
// M = 64, whose rows sit 16 to a TMEM lane quadrant -- and per page:
//   S = Q K^T       8 UMMA Mx128x16 -> TMEM S[buf] (fp32, lane = row)
//   softmax         warps 0-7: warp w reads TMEM lane quadrant w % 4 and
//                   columns 64 (w / 4) .. + 63 of its rows (M = 64: the
//                   16-lane load shape, two rows per thread; M = 128: one row
//                   per lane); the two warps of a quadrant swap their row
//                   maxima through shared memory.  Online maximum in the log2
//                   domain (O rescaled only when a row's maximum rises by more
//                   than 8; the stale maximum is exact since the final
//                   division uses the same one), P = 2^(x - m) as bf16 pairs
//                   stored back over S[buf]
//   O += P V        8 UMMA Mx128x16 with A = P in TMEM and B = the V page
//                   (token rows, MN-major, both 64-column halves in one
//                   instruction) -> TMEM O (fp32, 128 columns)
// Warp 8 streams Q (3-D box per sequence) and the K pages, warp 10 the V pages
// (two rings of 32 KB stages in the UMMA's 128B-swizzled layout, each stream
// as far ahead as its own ring allows), both with the pages' buffers looked up
// 32 to 64 pages ahead; warp 9 issues the UMMAs (one elected lane, four to a
// burst), QK of page i + 1 ahead of PV of page i so the tensor core overlaps
// the softmax (the last PV of a sequence is not held back).  TMEM: three S
// buffers at columns 0, 128, 256 and O at 384.
#pragma once

#include "attn.cuh"
#include "umma.cuh"

namespace trtv {

constexpr int kUmmaAttnThreads = 352;  // softmax warps 0-7, K/Q TMA 8, UMMA 9, V TMA 10
constexpr int kSBufs = 3;
constexpr uint32_t kAttnTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kQf8Tile = 64 * 128;  // FP8 caches: one E4M3 Q term, 64 rows x 128 B

// FP8 caches, E4M3 operands with two terms: x ~ hi + lo, hi = E4M3(x),
// lo = E4M3(x - hi) -- about 8 significant bits, as bf16 (one E4M3 term, 4
// bits, misses the 5e-2 output tolerance on rows that attend few positions).
// Two 16-bit values -> the hi and lo E4M3 pairs (low byte = first value).
__device__ __forceinline__ void split_e4m3x2(__half2 h, uint32_t& hi, uint32_t& lo) {
  __half2_raw hr = *reinterpret_cast<__half2_raw*>(&h);
  const __nv_fp8x2_storage_t h8 = __nv_cvt_halfraw2_to_fp8x2(hr, __NV_SATFINITE, __NV_E4M3);
  __half2_raw back = __nv_cvt_fp8x2_to_halfraw2(h8, __NV_E4M3);
  const __half2 rest = __hsub2(h, *reinterpret_cast<__half2*>(&back));
  __half2_raw rr = *reinterpret_cast<const __half2_raw*>(&rest);
  hi = h8;
  lo = __nv_cvt_halfraw2_to_fp8x2(rr, __NV_SATFINITE, __NV_E4M3);
}

// Row r of the bf16 Q tile (two 64-column halves, 128-byte swizzled) -> rows
// r of the hi and lo E4M3 Q tiles (one 128-byte row each, swizzled) for
// q / 2^e, 2^e the smallest power of two that brings max |q| of the row to at
// most 448 (dividing by it is exact).  Returns 2^e, the factor the row's
// logits are multiplied by.
__device__ __forceinline__ float quantize_q_row(const uint8_t* qb16, int half_bytes, uint8_t* qhi, uint8_t* qlo,
                                                int r) {
  const int sw = r & 7;
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < 16; ++c) {  // 16 chunks of 8 bf16: half c / 8, chunk c % 8
    const uint4 v = *reinterpret_cast<const uint4*>(qb16 + (c >> 3) * half_bytes + r * 128 + (((c & 7) ^ sw) << 4));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[k] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[k] & 0xFFFF0000u)));
    }
  }
  int e = 0;
  while (amax > 448.f * exp2f(static_cast<float>(e))) ++e;
  const float inv = exp2f(static_cast<float>(-e));
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {  // E4M3 chunk c8 = head dims 16 c8 .. + 15 = bf16 chunks 2 c8, 2 c8 + 1
    uint32_t oh[4], ol[4];
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const int c = 2 * c8 + part;
      const uint4 v = *reinterpret_cast<const uint4*>(qb16 + (c >> 3) * half_bytes + r * 128 + (((c & 7) ^ sw) << 4));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint32_t h0, l0, h1, l1;
        split_e4m3x2(__floats2half2_rn(__uint_as_float(w[2 * k] << 16) * inv,
                                       __uint_as_float(w[2 * k] & 0xFFFF0000u) * inv), h0, l0);
        split_e4m3x2(__floats2half2_rn(__uint_as_float(w[2 * k + 1] << 16) * inv,
                                       __uint_as_float(w[2 * k + 1] & 0xFFFF0000u) * inv), h1, l1);
        oh[2 * part + k] = (h0 & 0xFFFFu) | (h1 << 16);
        ol[2 * part + k] = (l0 & 0xFFFFu) | (l1 << 16);
      }
    }
    *reinterpret_cast<uint4*>(qhi + r * 128 + ((c8 ^ sw) << 4)) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
    *reinterpret_cast<uint4*>(qlo + r * 128 + ((c8 ^ sw) << 4)) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
  }
  return exp2f(static_cast<float>(e));
}

template <int D, bool FP8, bool SPREAD = false>
__global__ void __launch_bounds__(kUmmaAttnThreads, 1)
    attn_umma_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                     const __grid_constant__ AttnParams p) {
  static_assert(D == 128, "tcgen05 attention handles head_dim 128");
  // one page of K (or V) for one head: 32 KB of bf16, or 16 KB of E4M3 used as
  // it is by kind::f8f6f4 UMMAs (Q and P then also E4M3)
  constexpr int KV = FP8 ? kGroups * kBox : kGroups * 2 * kBox;
  // SPREAD (bf16 tiles of 33..64 rows): M = 64 UMMAs, whose accumulator (and
  // TMEM A operand) row m sits in lane 32 (m / 16) + m % 16: 16 rows in every
  // lane quadrant, so the softmax runs on all four SM sub-partitions (a warp
  // reaches only its own quadrant's lanes) at the cost of an M = 128 UMMA.
  static_assert(!(SPREAD && FP8), "the spread layout is for bf16 tiles");
  constexpr bool spread = SPREAD;
  const uint32_t IDESC_QK = FP8 ? umma_idesc_e4m3(128, 128) : umma_idesc_bf16(spread ? 64 : 128, 128);
  const uint32_t IDESC_PV = (FP8 ? umma_idesc_e4m3(128, 128) : umma_idesc_bf16(spread ? 64 : 128, 128)) |
                            (1u << 16);  // B (V) MN-major
  constexpr uint32_t TM_O = 384;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int NK = p.nstages, NV = p.nv, NQ = p.nq, QBUF = p.qbuf;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* kempty = kfull + NK;   // QK finished reading the K stage
  uint64_t* vfull = kempty + NK;
  uint64_t* vempty = vfull + NV;   // PV finished reading the V stage
  uint64_t* sfull = vempty + NV;        // [3] S written
  uint64_t* pfull = sfull + kSBufs;     // [3] P written over S (8 softmax warps)
  uint64_t* pvdone = pfull + kSBufs;    // [3] PV of the page in that buffer retired
  uint64_t* qfull = pvdone + kSBufs;    // [2]
  uint64_t* qempty = qfull + 2;    // [2] last QK of the sequence retired
  uint64_t* mdone = qempty + 2;
  // FP8: Q quantised to E4M3 (tile and per-row scales written), and the
  // softmax warps have read the row scales
  uint64_t* qcv = mdone + 1;       // [2]
  uint64_t* qsfree = qcv + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(qsfree + 1);
  int* abortf = reinterpret_cast<int*>(qsfree + 2);  // the CTA's give-up flag
  const Waits wt{p.err, abortf, p.wait_ns};
  int32_t* scan = reinterpret_cast<int32_t*>(smem + p.off_scan);
  // [0,256) merge flags, [256,512) merge row stats, [512,1024) row maxima of
  // the two column halves (double-buffered by page), [1024,1280) row sums
  float* ml = reinterpret_cast<float*>(smem + p.off_ml);
  const bool sparse = p.sparse != 0;
  const int Hk = p.num_kv_heads, T = p.qo_len, G = p.group;
  const int nitems = sparse ? p.batch * Hk : p.batch;
  int32_t* warp_tot = scan + nitems + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // softmax warps: all eight, or with FP8 those of lane quadrants holding
    // rows (the others quantise Q)
    const int live_quads = (G * T + 31) / 32;
    const int nsoft = FP8 ? 2 * live_quads : 8;
    for (int i = 0; i < NK; ++i) { mbar_init(&kfull[i], 1); mbar_init(&kempty[i], 1); }
    for (int i = 0; i < NV; ++i) { mbar_init(&vfull[i], 1); mbar_init(&vempty[i], 1); }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], nsoft);
      mbar_init(&pvdone[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
    }
    mbar_init(mdone, 1);
    *abortf = 0;
    if constexpr (FP8) {
      for (int i = 0; i < 2; ++i) mbar_init(&qcv[i], 8 - nsoft);
      mbar_init(qsfree, nsoft);
    }
    fence_mbar_init();
  }
  pdl_wait();  // inputs may come from the previous kernel of the stream
  block_exclusive_scan(nitems, scan, warp_tot, [&](int i) -> int32_t {
    return seq_units(p, i, T, sparse);
  });
  const int64_t W = item_start(scan, nitems, Hk, sparse);
  if (threadIdx.x == 0) write_split_desc(p, scan, nitems, Hk, sparse, W);
  pdl_trigger();  // the split-combine kernel may be scheduled now
  for (int i = blockIdx.x; i < nitems; i += gridDim.x) {  // zero rows of empty sequences
    if (scan[i + 1] != scan[i]) continue;
    const int b = sparse ? i / Hk : i;
    const int h0 = sparse ? i % Hk : 0, nh = sparse ? 1 : Hk;
    const int span = nh * G * D;
    for (int t = 0; t < T; ++t) {
      const int64_t o0 = ((static_cast<int64_t>(b) * T + t) * p.num_q_heads + static_cast<int64_t>(h0) * G) * D;
      for (int e = threadIdx.x; e < span; e += blockDim.x) {
        if (p.out_f32) static_cast<float*>(p.out)[o0 + e] = 0.f;
        else static_cast<__nv_bfloat16*>(p.out)[o0 + e] = __float2bfloat16(0.f);
      }
    }
  }
  if (W == 0) return;
  const int64_t u0 = cta_unit_begin(blockIdx.x, W, p.num_ctas);
  const int64_t u1 = cta_unit_begin(blockIdx.x + 1, W, p.num_ctas);
  if (u0 >= u1) return;

  // The small loads the first pages need go out now, ahead of the TMEM
  // allocation, the barrier below and the first wave of page copies: the
  // producers' page buffers of the first 64 pages, and the softmax warps'
  // plan entries and the first sequence's kv_len.
  const bool producer = warp == 8 || warp == 10;
  PageWalk pw{};
  PageAhead pa{};
  PlanAhead qa{};
  int Lc = 0;  // softmax warps: kv_len of the sequence about to start
  if (producer) {
    pw = walk_first(scan, nitems, Hk, sparse, u0, u1, p.setup);
    ahead_init(pa, p, pw, lane, sparse, warp == 10, scan, nitems, Hk, u0, u1);
  } else if (warp < 8) {
    if (sparse) plan_ahead_init(qa, p, lane, scan, nitems, Hk, u0, u1);
    Lc = p.kv_lens[cursor_first(scan, nitems, Hk, sparse, u0).b];
  }
  if (warp == 9) {
    tmem_alloc(tslot, kAttnTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  uint8_t* qbase = smem + p.off_q;
  uint8_t* kring = smem + p.off_stage;
  uint8_t* vring = smem + p.off_vring;
  uint8_t* qf8 = smem + p.off_qf8;   // FP8: E4M3 Q tile, [rows][128 B], 128-byte swizzled
  float* qscale = reinterpret_cast<float*>(smem + p.off_ml);  // FP8: [128] per-row Q scales

  if (producer) {
    // ------------------------------------------- TMA producers: K (+Q) and V
    // Two independent streams: K pages are freed early (after QK), V pages
    // late (after PV); one stream must not hold the other back.  The pages'
    // buffers come from the page-ahead groups (one page per lane, resolved 32
    // to 64 pages early); lane 0 waits and issues.
    const bool is_v = warp == 10;
    if (lane == 0) {
      prefetch_tensormap(&kv_map);
      if (!is_v) prefetch_tensormap(&q_map);
    }
    const uint64_t pol = policy_evict_first();
    const int sub_rows = Hk * kSub;
    const uint32_t qbytes = static_cast<uint32_t>(2 * 64 * 2 * G * T);
    const int n = is_v ? NV : NK;
    uint64_t* fullb = is_v ? vfull : kfull;
    uint64_t* emptyb = is_v ? vempty : kempty;
    uint8_t* ring = is_v ? vring : kring;
    int it = 0, sq = 0, st = 0;
    uint32_t eph = 1;  // parity of the empty-barrier phase that frees stage st
    PageWalk w = pw;
    while (w.valid) {
      if (!is_v && w.j == w.j0) {  // a sequence starts: its Q tile first
        const int qb = sq % NQ;
        bool ok = true;
        if (lane == 0 && sq >= NQ) ok = mbar_wait(&qempty[qb], static_cast<uint32_t>(sq / NQ - 1) & 1u, wt);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&qfull[qb], qbytes);
          for (int hb = 0; hb < 2; ++hb)
            asm volatile(
                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(qbase + qb * QBUF + hb * (QBUF / 2))),
                "l"(reinterpret_cast<uint64_t>(&q_map)), "r"(hb * 64), "r"(w.cur.h * G), "r"(w.cur.b * T),
                "r"(smem_u32(&qfull[qb]))
                : "memory");
        }
        ++sq;
      }
      if (!is_v && p.withhold >= 0 && it >= p.withhold) break;  // tests of the give-up path only
      int spe[kGroups];
#pragma unroll
      for (int g = 0; g < kGroups; ++g) spe[g] = __shfl_sync(0xffffffffu, pa.now[g], it & 31);
      page_buffers(p, is_v, !is_v, spe);
      bool ok = true;
      if (lane == 0 && it >= n) ok = mbar_wait(&emptyb[st], eph, wt);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) {
        uint8_t* dst = ring + st * KV;
        mbar_arrive_expect_tx(&fullb[st], KV);
        // bf16: two 128-byte column halves per sub-page; FP8: one box holds
        // all 128 head dims of a token row
#pragma unroll
        for (int hb = 0; hb < (FP8 ? 1 : 2); ++hb)
#pragma unroll
          for (int g = 0; g < kGroups; ++g)
            tma_load_2d(dst + (hb * kGroups + g) * kBox, &kv_map, &fullb[st], hb * 64,
                        spe[g] * sub_rows + w.cur.h * kSub, pol);
      }
      if (++st == n) {
        st = 0;
        eph ^= 1u;
      }
      ++it;
      walk_skip(w, 1, scan, nitems, Hk, sparse, u0, u1, p.setup);
      if ((it & 31) == 0) ahead_step(pa, p, lane, sparse, is_v, scan, nitems, Hk, u0, u1);
    }
    // never leave copies in flight
    if (lane == 0) {
      for (int k = (it > n ? it - n : 0); k < it; ++k)
        mbar_drain(&fullb[k % n], static_cast<uint32_t>(k / n) & 1u, wt);
      if (!is_v && sq >= 1)
        mbar_drain(&qfull[(sq - 1) % NQ], static_cast<uint32_t>((sq - 1) / NQ) & 1u, wt);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ----------------------------------------------------------- UMMA issuer
    // The whole warp runs the loop (uniform control flow, operands in uniform
    // registers) and one elected lane issues; lane 0 waits for the barriers.
    // Descriptors are built once and moved by byte offsets; ring positions
    // advance by increments (no division in the loop).
    const uint64_t kd0 = umma_desc_sw128(smem_u32(kring));
    const uint64_t qd0 = umma_desc_sw128(smem_u32(FP8 ? qf8 : qbase));
    const uint64_t vd0 = FP8 ? umma_desc_sw128_lbo_sbo(smem_u32(vring), 1024, 1024)
                             : umma_desc_sw128_mn(smem_u32(vring), KV / 2);
    auto wait1 = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, lane != 0 || mbar_wait(bar, par, wt));
    };
    bool alive = true;
    int ks = 0, vs = 0, sb = 0, pb = 0, qb = 0;
    uint32_t kph = 0, vph = 0, sph = 0, pph = 0, qph = 0;
    int it = 0;
    // O += P V for the next page in PV order (S buffer pb, V stage vs);
    // `first`: the sequence's first page (O starts over)
    auto issue_pv = [&](bool first) {
      if (!alive) return;
      if (!wait1(&vfull[vs], vph) || !wait1(&pfull[pb], pph)) {
        alive = false;
        return;
      }
      tc_fence_after();
      const uint64_t va = desc_add(vd0, static_cast<uint32_t>(vs * KV));
      const uint32_t pa = tmem + static_cast<uint32_t>(pb * 128);
      // FP8: 32 tokens (8 P columns, 32 V rows of 128 B = 4 KB) per UMMA, all
      // 128 head dims one swizzle atom, O += P_hi V + P_lo V (P_hi in columns
      // 0..31, P_lo in 32..63).  bf16: 16 tokens per UMMA, both 64-column
      // halves of V in one instruction.
#pragma unroll
      for (int h4 = 0; h4 < 2; ++h4) {
        uint32_t a[4];
        uint64_t b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          a[i] = FP8 ? pa + h4 * 32 + i * 8 : pa + (4 * h4 + i) * 8;
          b[i] = desc_add(va, FP8 ? i * 4096 : (4 * h4 + i) * 2048);
        }
        umma4_tmem_a_elect<FP8>(tmem + TM_O, a, b, IDESC_PV, (!first || h4 > 0) ? 1u : 0u);
      }
      umma_commit_elect(&vempty[vs]);
      umma_commit_elect(&pvdone[pb]);
      if (++vs == NV) {
        vs = 0;
        vph ^= 1u;
      }
      if (++pb == kSBufs) {
        pb = 0;
        pph ^= 1u;
      }
    };
    bool pend = false, pend_first = false;
    for (SeqCursor cur = cursor_first(scan, nitems, Hk, sparse, u0);
         alive && (sparse ? cur.s : cur.b) < nitems && seq_in_range(cur, u1, p.setup);
         cursor_next(cur, scan, nitems, Hk, sparse)) {
      if (!wait1(FP8 ? &qcv[qb] : &qfull[qb], qph)) {
        alive = false;
        break;
      }
      const uint64_t qd = desc_add(qd0, static_cast<uint32_t>(FP8 ? 0 : qb * QBUF));
      const int64_t j0 = seq_j0(cur, u0, p.setup), j1 = seq_j1(cur, u1, p.setup);
      for (int64_t j = j0; j < j1 && alive; ++j, ++it) {
        // S buffer sb was last read by the PV of page it - 3
        if (!wait1(&kfull[ks], kph) || (it >= kSBufs && !wait1(&pvdone[sb], sph ^ 1u))) {
          alive = false;
          break;
        }
        tc_fence_after();
        const uint64_t ka = desc_add(kd0, static_cast<uint32_t>(ks * KV));
        // FP8: a 128-byte row holds all 128 head dims, K = 32 per UMMA,
        // S = Q_hi K^T + Q_lo K^T.  bf16: K = 16, the head dims' two 64-column
        // halves KV / 2 (K page) and QBUF / 2 (Q tile) apart.
#pragma unroll
        for (int h4 = 0; h4 < 2; ++h4) {
          uint64_t a[4], b[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a[i] = desc_add(qd, FP8 ? h4 * kQf8Tile + i * 32 : h4 * (QBUF / 2) + i * 32);
            b[i] = desc_add(ka, FP8 ? i * 32 : h4 * (KV / 2) + i * 32);
          }
          umma4_elect<FP8>(tmem + static_cast<uint32_t>(sb * 128), a, b, IDESC_QK, h4 > 0 ? 1u : 0u);
        }
        umma_commit_elect(&kempty[ks]);
        umma_commit_elect(&sfull[sb]);
        if (j == j1 - 1) umma_commit_elect(&qempty[qb]);
        if (++ks == NK) {
          ks = 0;
          kph ^= 1u;
        }
        if (++sb == kSBufs) {
          sb = 0;
          sph ^= 1u;
        }
        if (pend) issue_pv(pend_first);
        pend = true;
        pend_first = j == j0;
      }
      // the sequence's last PV goes out now: its epilogue must not wait for
      // the next sequence's Q tile and first QK
      if (pend) issue_pv(pend_first);
      pend = false;
      if (++qb == NQ) {
        qb = 0;
        qph ^= 1u;
      }
    }
    umma_commit_elect(mdone);
    if (lane == 0) mbar_drain(mdone, 0, wt);
    __syncwarp();
  } else {
    // -------------------------------------------------- softmax and epilogue
    const int q = warp & 3;            // TMEM lane quadrant
    const int hf = warp >> 2;          // column half of every row
    if (FP8 && 32 * q >= G * T) {  // (a constant false for bf16 caches)
      // ------------------------------------------- FP8: Q quantiser warps
      // The softmax warps of lane quadrants without rows turn each sequence's
      // bf16 Q tile into the E4M3 tile the QK UMMA reads, one thread per row,
      // with a power-of-two scale per row that the softmax applies to the
      // row's logits.  The row scales have one slot: a sequence's scales are
      // written only after the softmax warps have read the previous ones.
      const int live_quads = (G * T + 31) / 32, nconv = 8 - 2 * live_quads;
      const int ct = ((q - live_quads) * 2 + hf) * 32 + lane, nct = nconv * 32;
      bool dead = false;
      int sq = 0;
      for (SeqCursor cur = cursor_first(scan, nitems, Hk, sparse, u0);
           (sparse ? cur.s : cur.b) < nitems && seq_in_range(cur, u1, p.setup);
           cursor_next(cur, scan, nitems, Hk, sparse), ++sq) {
        const int qb = sq % NQ;
        if (!dead)
          dead = __any_sync(0xffffffffu, !mbar_wait(&qfull[qb], static_cast<uint32_t>(sq / NQ) & 1u, wt));
        if (!dead && sq >= 1)
          dead = __any_sync(0xffffffffu, !mbar_wait(qsfree, static_cast<uint32_t>(sq - 1) & 1u, wt));
        for (int r = ct; r < G * T; r += nct)
          qscale[r] = quantize_q_row(qbase + qb * QBUF, QBUF / 2, qf8, qf8 + kQf8Tile, r);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&qcv[qb]);
      }
    } else if (SPREAD) {
      // --------------------------- softmax and epilogue, 64-row bf16 tiles
      // Rows 16q .. 16q + 15 sit in TMEM lanes 32q .. 32q + 15.  The 16-lane
      // load shape gives thread t two rows, ra = 16q + t / 4 and rb = ra + 8,
      // and of every 8-column chunk the columns 2 (t % 4) and + 1, so all 32
      // threads of the warp hold live values; a row's four threads reduce its
      // maximum and sum with two shuffles.  P goes back with the 16x128b
      // shape: the positions 2c, 2c + 1 a thread holds are exactly packed P
      // column c of its rows.
      const int g4 = lane >> 2, u4 = lane & 3;
      const int ra = 16 * q + g4, rb = ra + 8;
      const int ta = ra / G, tb = rb / G;
      const bool va = ta < T, vb = tb < T;
      const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
      float* xmax = ml + 512;  // [2 pages][2 halves][128 rows]
      float* xl = ml + 1024;   // [2 halves][128 rows]
      bool dead = false;
      int it = 0;
      for (SeqCursor cur = cursor_first(scan, nitems, Hk, sparse, u0);
           (sparse ? cur.s : cur.b) < nitems && seq_in_range(cur, u1, p.setup);
           cursor_next(cur, scan, nitems, Hk, sparse)) {
        const int L = Lc;
        {  // the next sequence's kv_len loads a whole sequence ahead of its use
          SeqCursor nx = cur;
          cursor_next(nx, scan, nitems, Hk, sparse);
          if ((sparse ? nx.s : nx.b) < nitems) Lc = p.kv_lens[nx.b];
        }
        const int bound_a = va ? L - T + ta : -1, bound_b = vb ? L - T + tb : -1;
        const int64_t j0 = seq_j0(cur, u0, p.setup), j1 = seq_j1(cur, u1, p.setup);
        const float scale = p.scale_log2;
        float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
        for (int64_t j = j0; j < j1; ++j, ++it) {
          const int buf = it % kSBufs;
          int blk = static_cast<int>(j);
          uint32_t tokmask = 0xffffffffu;
          if (sparse) {  // the page's plan entry, loaded 32 to 64 pages ahead
            if (it > 0 && (it & 31) == 0) plan_ahead_step(qa, p, lane, scan, nitems, Hk, u0, u1);
            blk = __shfl_sync(0xffffffffu, qa.blk_now, it & 31);
            tokmask = __shfl_sync(0xffffffffu, qa.m_now, it & 31);
          }
          if (!dead)
            dead = __any_sync(0xffffffffu, !mbar_wait(&sfull[buf], static_cast<uint32_t>(it / kSBufs) & 1u, wt));
          tc_fence_after();
          const int pos0 = blk * kPage + hf * 64 + 2 * u4;  // this thread's first position
          const int bnda = (va && ((tokmask >> ta) & 1u)) ? bound_a : -1;
          const int bndb = (vb && ((tokmask >> tb) & 1u)) ? bound_b : -1;
          const bool masked = sparse || blk * kPage + kPage - 1 > L - T;
          uint32_t sv[32];
          tmem_ld16x256_x8(tl + buf * 128 + hf * 64, sv);
          tmem_ld_wait_dep(sv);
          float xa[16], xb[16];
          float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
          for (int k = 0; k < 8; ++k)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int pos = pos0 + 8 * k + e;
              float a = __uint_as_float(sv[4 * k + e]) * scale;
              float b = __uint_as_float(sv[4 * k + 2 + e]) * scale;
              if (masked && pos > bnda) a = -INFINITY;
              if (masked && pos > bndb) b = -INFINITY;
              xa[2 * k + e] = a;
              xb[2 * k + e] = b;
              mxa = fmaxf(mxa, a);
              mxb = fmaxf(mxb, b);
            }
          mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
          mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
          mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
          mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
          if (u4 == 0) {
            xmax[((it & 1) * 2 + hf) * 128 + ra] = mxa;
            xmax[((it & 1) * 2 + hf) * 128 + rb] = mxb;
          }
          named_barrier(2 + q, 64);
          mxa = fmaxf(mxa, xmax[((it & 1) * 2 + (hf ^ 1)) * 128 + ra]);
          mxb = fmaxf(mxb, xmax[((it & 1) * 2 + (hf ^ 1)) * 128 + rb]);
          const float mna = fmaxf(ma, mxa), mnb = fmaxf(mb, mxb);
          const bool needa = ma != -INFINITY && mna > ma + kRescaleLog2;
          const bool needb = mb != -INFINITY && mnb > mb + kRescaleLog2;
          if (ma == -INFINITY) ma = mna;
          if (mb == -INFINITY) mb = mnb;
          if (__any_sync(0xffffffffu, needa || needb)) {
            // O must be stable: PV of the previous page has retired
            const int pv = it - 1;
            if (!dead)
              dead = __any_sync(0xffffffffu,
                                !mbar_wait(&pvdone[pv % kSBufs], static_cast<uint32_t>(pv / kSBufs) & 1u, wt));
            tc_fence_after();
            const float aa = needa ? fast_exp2(ma - mna) : 1.f, ab = needb ? fast_exp2(mb - mnb) : 1.f;
            if (needa) {
              la *= aa;
              ma = mna;
            }
            if (needb) {
              lb *= ab;
              mb = mnb;
            }
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
              uint32_t w[16];
              tmem_ld16x256_x4(tl + TM_O + hf * 64 + c0, w);
              tmem_ld_wait_dep(w);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                w[4 * k] = __float_as_uint(__uint_as_float(w[4 * k]) * aa);
                w[4 * k + 1] = __float_as_uint(__uint_as_float(w[4 * k + 1]) * aa);
                w[4 * k + 2] = __float_as_uint(__uint_as_float(w[4 * k + 2]) * ab);
                w[4 * k + 3] = __float_as_uint(__uint_as_float(w[4 * k + 3]) * ab);
              }
              tmem_st16x256_x4(tl + TM_O + hf * 64 + c0, w);
            }
            tmem_st_wait();
          }
          const bool nonea = ma == -INFINITY, noneb = mb == -INFINITY;
          uint32_t pw[16];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float a0 = nonea ? 0.f : fast_exp2(xa[2 * k] - ma);
            const float a1 = nonea ? 0.f : fast_exp2(xa[2 * k + 1] - ma);
            const float b0 = noneb ? 0.f : fast_exp2(xb[2 * k] - mb);
            const float b1 = noneb ? 0.f : fast_exp2(xb[2 * k + 1] - mb);
            la += a0 + a1;
            lb += b0 + b1;
            __nv_bfloat162 pa2 = __floats2bfloat162_rn(a0, a1), pb2 = __floats2bfloat162_rn(b0, b1);
            pw[2 * k] = *reinterpret_cast<uint32_t*>(&pa2);
            pw[2 * k + 1] = *reinterpret_cast<uint32_t*>(&pb2);
          }
          tmem_st16x128_x8(tl + buf * 128 + hf * 32, pw);
          tmem_st_wait();
          // V rows at or past kv_len may hold anything (NaN included): P is
          // zero there, but 0 * NaN is not, so warp 0 zeroes them first.
          const int nvalid = L - blk * kPage;
          if (warp == 0 && nvalid < kPage) {
            const int vs = it % NV;
            if (!dead)
              dead = __any_sync(0xffffffffu, !mbar_wait(&vfull[vs], static_cast<uint32_t>(it / NV) & 1u, wt));
            uint8_t* vst = vring + vs * KV;
            const int nchunks = (kPage - nvalid) * 16;
            for (int idx = lane; idx < nchunks; idx += 32) {
              const int tok = nvalid + idx / 16, part = idx % 16;
              *reinterpret_cast<uint4*>(vst + ((part >> 3) * kGroups + tok / kSub) * kBox + (tok % kSub) * 128 +
                                        (part & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&pfull[buf]);
        }
        // ----------------------------------------------------- sequence end
        const int last = it - 1;
        if (!dead)
          dead = __any_sync(0xffffffffu,
                            !mbar_wait(&pvdone[last % kSBufs], static_cast<uint32_t>(last / kSBufs) & 1u, wt));
        tc_fence_after();
        const bool whole = seq_whole(cur, u0, u1, p.setup);
        const int64_t slot = seq_slot(cur, u0, p.setup);
        la += __shfl_xor_sync(0xffffffffu, la, 1);
        lb += __shfl_xor_sync(0xffffffffu, lb, 1);
        la += __shfl_xor_sync(0xffffffffu, la, 2);
        lb += __shfl_xor_sync(0xffffffffu, lb, 2);
        if (u4 == 0) {
          xl[hf * 128 + ra] = la;
          xl[hf * 128 + rb] = lb;
        }
        named_barrier(2 + q, 64);
        const float lta = la + xl[(hf ^ 1) * 128 + ra], ltb = lb + xl[(hf ^ 1) * 128 + rb];
        const float inva = lta > 0.f ? 1.f / lta : 0.f, invb = ltb > 0.f ? 1.f / ltb : 0.f;
        const float sca = whole ? inva * p.v_scale : inva, scb = whole ? invb * p.v_scale : invb;
        uint32_t ov[32];
        tmem_ld16x256_x8(tl + TM_O + hf * 64, ov);
        tmem_ld_wait_dep(ov);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {  // rows ra, rb
          const int row = h2 ? rb : ra, tt = h2 ? tb : ta;
          const float sc = h2 ? scb : sca;
          if (!(h2 ? vb : va)) continue;
          const int64_t orow = ((static_cast<int64_t>(cur.b) * T + tt) * p.num_q_heads +
                                static_cast<int64_t>(cur.h) * G + row % G) * D + hf * 64 + 2 * u4;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float o0 = __uint_as_float(ov[4 * k + 2 * h2]) * sc;
            const float o1 = __uint_as_float(ov[4 * k + 2 * h2 + 1]) * sc;
            if (whole) {
              if (p.out_f32) {
                *reinterpret_cast<float2*>(static_cast<float*>(p.out) + orow + 8 * k) = make_float2(o0, o1);
              } else {
                __nv_bfloat162 pk = __floats2bfloat162_rn(o0, o1);
                *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + orow + 8 * k) = pk;
              }
            } else {
              *reinterpret_cast<float2*>(p.ws_o + (slot * p.rows_pad + row) * D + hf * 64 + 2 * u4 + 8 * k) =
                  make_float2(o0, o1);
            }
          }
          if (!whole && hf == 0 && u4 == 0) {
            const float lt = h2 ? ltb : lta, m = h2 ? mb : ma;
            p.ws_lse[slot * p.rows_pad + row] = lt > 0.f ? m + __log2f(lt) : -INFINITY;
          }
        }
        tc_fence_before();
      }
    } else {
    const int r = 32 * q + lane;                                   // this thread's TMEM lane
    const int row = spread ? (lane < 16 ? 16 * q + lane : 1 << 20) : r;  // its (token, group head) row
    const int t = row / G, gl = row % G;
    const bool valid = t < T;
    const bool live = spread || 32 * q < G * T;  // same for both warps of a quadrant
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
    float* xmax = ml + 512;            // [2 pages][2 halves][128 rows]
    float* xl = ml + 1024;             // [2 halves][128 rows]
    bool dead = false;
    int it = 0, sq = 0;
    for (SeqCursor cur = cursor_first(scan, nitems, Hk, sparse, u0);
         (sparse ? cur.s : cur.b) < nitems && seq_in_range(cur, u1, p.setup);
         cursor_next(cur, scan, nitems, Hk, sparse), ++sq) {
      const int L = Lc;
      {  // the next sequence's kv_len loads a whole sequence ahead of its use
        SeqCursor nx = cur;
        cursor_next(nx, scan, nitems, Hk, sparse);
        if ((sparse ? nx.s : nx.b) < nitems) Lc = p.kv_lens[nx.b];
      }
      const int bound = valid ? L - T + t : -1;
      const int64_t j0 = seq_j0(cur, u0, p.setup), j1 = seq_j1(cur, u1, p.setup);
      float m_use = -INFINITY, l = 0.f;
      // logit scale in the log2 domain; FP8: times the row's Q scale
      float scale = p.scale_log2;
      if constexpr (FP8) {
        if (!dead)
          dead = __any_sync(0xffffffffu, !mbar_wait(&qcv[sq % NQ], static_cast<uint32_t>(sq / NQ) & 1u, wt));
        scale *= valid ? qscale[r] : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(qsfree);
      }
      for (int64_t j = j0; j < j1; ++j, ++it) {
        const int buf = it % kSBufs;
        int blk = static_cast<int>(j);
        uint32_t tokmask = 0xffffffffu;
        if (sparse) {  // the page's plan entry, loaded 32 to 64 pages ahead
          if (it > 0 && (it & 31) == 0) plan_ahead_step(qa, p, lane, scan, nitems, Hk, u0, u1);
          blk = __shfl_sync(0xffffffffu, qa.blk_now, it & 31);
          tokmask = __shfl_sync(0xffffffffu, qa.m_now, it & 31);
        }
        if (!dead)
          dead = __any_sync(0xffffffffu, !mbar_wait(&sfull[buf], static_cast<uint32_t>(it / kSBufs) & 1u, wt));
        tc_fence_after();
        const int pos0 = blk * kPage;
        if (live) {
          const int bnd = (valid && ((tokmask >> t) & 1u)) ? bound : -1;
          const bool masked = sparse || pos0 + kPage - 1 > L - T;
          uint32_t ra[32], rb[32];
          tmem_ld32_async(tl + buf * 128 + hf * 64, ra);
          tmem_ld32_async(tl + buf * 128 + hf * 64 + 32, rb);
          tmem_ld_wait_dep(ra);
          tmem_ld_wait_dep(rb);
          float x[64];
          float mloc = -INFINITY;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            float v = __uint_as_float(i < 32 ? ra[i] : rb[i - 32]) * scale;
            if (masked && pos0 + hf * 64 + i > bnd) v = -INFINITY;
            x[i] = v;
            mloc = fmaxf(mloc, v);
          }
          xmax[((it & 1) * 2 + hf) * 128 + r] = mloc;
          named_barrier(2 + q, 64);
          mloc = fmaxf(mloc, xmax[((it & 1) * 2 + (hf ^ 1)) * 128 + r]);
          const float m_new = fmaxf(m_use, mloc);
          const bool need = m_use != -INFINITY && m_new > m_use + kRescaleLog2;
          if (m_use == -INFINITY) m_use = m_new;
          if (__any_sync(0xffffffffu, need)) {
            // O must be stable: PV of the previous page has retired
            const int pv = it - 1;
            if (!dead)
              dead = __any_sync(0xffffffffu, !mbar_wait(&pvdone[pv % kSBufs], static_cast<uint32_t>(pv / kSBufs) & 1u, wt));
            tc_fence_after();
            const float alpha = need ? fast_exp2(m_use - m_new) : 1.f;
            if (need) {
              l *= alpha;
              m_use = m_new;
            }
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {  // 16 columns at a time: x[] stays live meanwhile
              uint32_t w[16];
              tmem_ld_async(tl + TM_O + hf * 64 + c0, w);
              tmem_ld_wait_dep(w);
#pragma unroll
              for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
              tmem_st16(tl + TM_O + hf * 64 + c0, w);
            }
            tmem_st_wait();
          }
          const bool none = m_use == -INFINITY;
          if constexpr (FP8) {
            // P = P_hi + P_lo as E4M3, four positions per TMEM column (P is at
            // most 2^8 < 448: the reference maximum lags by at most 8); l sums
            // the fp32 values
            uint32_t wh[16], wl[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float pv[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                pv[k] = none ? 0.f : fast_exp2(x[4 * i + k] - m_use);
                l += pv[k];
              }
              uint32_t h0, l0, h1, l1;
              split_e4m3x2(__floats2half2_rn(pv[0], pv[1]), h0, l0);
              split_e4m3x2(__floats2half2_rn(pv[2], pv[3]), h1, l1);
              wh[i] = (h0 & 0xFFFFu) | (h1 << 16);
              wl[i] = (l0 & 0xFFFFu) | (l1 << 16);
            }
            tmem_st16(tl + buf * 128 + hf * 16, wh);
            tmem_st16(tl + buf * 128 + 32 + hf * 16, wl);
          } else {
            // two halves of 16 columns: fewer values live at once
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t w[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float p0 = none ? 0.f : fast_exp2(x[32 * h2 + 2 * i] - m_use);
                const float p1 = none ? 0.f : fast_exp2(x[32 * h2 + 2 * i + 1] - m_use);
                l += p0 + p1;
                __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
                w[i] = *reinterpret_cast<uint32_t*>(&pk);
              }
              tmem_st16(tl + buf * 128 + hf * 32 + 16 * h2, w);
            }
          }
          tmem_st_wait();
        }
        // V rows at or past kv_len may hold anything (NaN included): P is zero
        // there, but 0 * NaN is not, so warp 0 zeroes them before PV reads V.
        const int nvalid = L - pos0;
        if (warp == 0 && nvalid < kPage) {
          const int vs = it % NV;
          if (!dead)
            dead = __any_sync(0xffffffffu, !mbar_wait(&vfull[vs], static_cast<uint32_t>(it / NV) & 1u, wt));
          uint8_t* vst = vring + vs * KV;
          constexpr int NHALF = FP8 ? 1 : 2;  // 128-byte column blocks per token row
          const int nchunks = (kPage - nvalid) * 8 * NHALF;
          for (int idx = lane; idx < nchunks; idx += 32) {
            const int tok = nvalid + idx / (8 * NHALF), part = idx % (8 * NHALF);
            *reinterpret_cast<uint4*>(vst + ((part >> 3) * kGroups + tok / kSub) * kBox + (tok % kSub) * 128 +
                                      (part & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[buf]);
      }
      // ------------------------------------------------------- sequence end
      const int last = it - 1;
      if (!dead)
        dead = __any_sync(0xffffffffu, !mbar_wait(&pvdone[last % kSBufs], static_cast<uint32_t>(last / kSBufs) & 1u, wt));
      tc_fence_after();
      const bool whole = seq_whole(cur, u0, u1, p.setup);
      const int64_t slot = seq_slot(cur, u0, p.setup);
      if (live) {
        xl[hf * 128 + r] = l;
        named_barrier(2 + q, 64);
        const float lt = l + xl[(hf ^ 1) * 128 + r];
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const float sc = whole ? inv * p.v_scale : inv;
        const int64_t orow = ((static_cast<int64_t>(cur.b) * T + t) * p.num_q_heads +
                              static_cast<int64_t>(cur.h) * G + gl) * D + hf * 64;
        uint32_t oa[32], ob[32];
        tmem_ld32_async(tl + TM_O + hf * 64, oa);
        tmem_ld32_async(tl + TM_O + hf * 64 + 32, ob);
        tmem_ld_wait_dep(oa);
        tmem_ld_wait_dep(ob);
        if (valid) {
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            const uint32_t* v = c0 ? ob : oa;
            if (whole) {
              if (p.out_f32) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow + c0);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  dst[i] = make_float4(__uint_as_float(v[4 * i]) * sc, __uint_as_float(v[4 * i + 1]) * sc,
                                       __uint_as_float(v[4 * i + 2]) * sc, __uint_as_float(v[4 * i + 3]) * sc);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow + c0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  uint32_t w4[4];
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    __nv_bfloat162 pk = __floats2bfloat162_rn(__uint_as_float(v[8 * i + 2 * k]) * sc,
                                                              __uint_as_float(v[8 * i + 2 * k + 1]) * sc);
                    w4[k] = *reinterpret_cast<uint32_t*>(&pk);
                  }
                  dst[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
              }
            } else {
              float4* dst = reinterpret_cast<float4*>(p.ws_o + (slot * p.rows_pad + row) * D + hf * 64 + c0);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(__uint_as_float(v[4 * i]) * sc, __uint_as_float(v[4 * i + 1]) * sc,
                                     __uint_as_float(v[4 * i + 2]) * sc, __uint_as_float(v[4 * i + 3]) * sc);
            }
          }
          if (!whole && hf == 0) p.ws_lse[slot * p.rows_pad + row] = lt > 0.f ? m_use + __log2f(lt) : -INFINITY;
        }
      }
      tc_fence_before();
    }
    }  // softmax warps
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kAttnTmemCols);
  }
}

}  // namespace trtv
