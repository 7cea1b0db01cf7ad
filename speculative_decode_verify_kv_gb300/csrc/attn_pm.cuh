// attn_pm.cuh -- ladder verify attention (dense and MSA sparse) on the
// tcgen05 tensor cores with the page's 128 positions as the UMMA's M and the
// (token, group head) rows as its N ("position-major"), for tiles of at most
// 32 rows: FP8 E4M3 K/V (the library instantiates it for FP8 caches; the
// template also takes bf16), head_dim 128, G = Hq / Hk a power of two.
//
// Sources: "Eagle3 for M3 MSA path + CUDA graphs compatibility" (fork PR #3),
// commit "... verify" (token t attends kv_len - qo_len + t + 1 positions; the
// sparse pass attends the selected blocks); "Default Minimax-m3 to unified
// draft-target kv manager" (#17835), "Grouped-HND draft KV transfer" (page
// layout); "wrap up eagle changes in m3 side branch" (#18066), view commit
// (K page at slot * stride, V page at slot * stride + 1).
//
// A tcgen05.mma costs its issue slot whatever its N: small row tiles as M
// would fill a fraction of each instruction, while the positions as M keep
// all 128 lanes busy and the count of instructions per page is the same.
// Per (request, KV head) sequence the rows c = t * G + g are the N columns
// (NR = 16 or 32 rows; with FP8 caches the hi and lo E4M3 terms of Q and P
// are the two halves of N = 2 NR, so one instruction covers both), and per
// page:
//   S^T = K Q^T     A = the K page (positions x head dims, K-major as TMA
//                   stages it), B = the Q tile (rows x head dims, K-major):
//                   8 bf16 UMMA 128 x NR x 16, or 4 E4M3 UMMA 128 x 2NR x 32
//                   -> TMEM S[it % 2] (lane = position, column = row)
//   softmax         NR / 2 warps: warp w reads TMEM lane quadrant w % 4 (32
//                   positions) and the 8 columns 8 (w / 4) .. + 7.  A column's
//                   reference maximum moves only when a value exceeds it by
//                   more than 8 (log2 domain): the four quadrant warps vote,
//                   and only on a "yes" (always on a sequence's first page)
//                   are the exact column maxima exchanged -- a lane
//                   transpose-reduction and shared memory -- and O^T
//                   rescaled where a maximum rose by more than 8; P^T =
//                   2^(x - m) written to shared memory as bf16, or as two
//                   E4M3 terms (P < 2^8 fits E4M3)
//   O^T += V^T P^T  A = the V page read MN-major (head dims x positions), B =
//                   P^T MN-major (rows x positions): 8 bf16 UMMA 128 x NR x 16
//                   or 4 E4M3 UMMA 128 x 2NR x 32 -> TMEM O^T (lane = head dim)
// Pages go through the QK, softmax and PV stages in pairs (of one sequence):
// the softmax takes both pages of a pair in one pass -- one wait, one vote,
// one barrier and one arrival per pair, and twice the independent arithmetic
// between them.  After the softmax warps: one warp streams Q and the K pages,
// one issues the UMMAs (one elected lane; QK of pair i + 1 ahead of PV of pair
// i), one streams the V pages (rings of 32 KB bf16 or 16 KB E4M3 stages), and
// with FP8 caches one turns each sequence's bf16 Q tile into the two E4M3
// terms with a power-of-two scale per row.  P^T buffers live in 16 KB regions
// of 128-byte rows, 2 NR bytes each (bf16: NR values; E4M3: NR hi bytes then
// NR lo bytes).  TMEM: four S^T buffers (two pair slots) and O^T, each N
// columns wide.
#pragma once

#include "attn.cuh"
#include "attn_umma.cuh"
#include "umma.cuh"

namespace trtv {

// Warps: 4 NR / 8 softmax warps (one per TMEM lane quadrant and group of 8
// columns), then the K/Q TMA producer, the UMMA issuer, the V TMA producer and
// (FP8 caches) the Q quantiser.
__host__ __device__ constexpr int pm_softmax_warps(int nr) { return nr / 2; }
__host__ __device__ constexpr int pm_threads(bool fp8, int nr) { return (pm_softmax_warps(nr) + (fp8 ? 4 : 3)) * 32; }
constexpr int kPmPRegion = 128 * 128;  // P^T buffers: 128 rows of 128 B

// Reduction across the 32 lanes of a warp of H values per lane, value i
// belonging to column i: afterwards lane l holds the result for column
// l >> (5 - log2 H).  log2 H exchange steps each hand half of the remaining
// columns to the partner lane (a transpose-reduction), then the lanes that
// share a column combine.  v is destroyed.
template <int H, bool MAX>
__device__ __forceinline__ float lane_col_reduce(float (&v)[H], int lane) {
  constexpr int LH = H == 8 ? 3 : (H == 16 ? 4 : 5);
  static_assert((1 << LH) == H, "8, 16 or 32 columns");
#pragma unroll
  for (int s = 0; s < LH; ++s) {
    const int m = 16 >> s;
    const int n = H >> (s + 1);
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < (H >> 1); ++i) {
      if (i < n) {
        const float send = up ? v[i] : v[i + n];
        const float keep = up ? v[i + n] : v[i];
        const float got = __shfl_xor_sync(0xffffffffu, send, m);
        v[i] = MAX ? fmaxf(keep, got) : keep + got;
      }
    }
  }
  float r = v[0];
#pragma unroll
  for (int m = 1; m < (1 << (5 - LH)); m <<= 1) {
    const float got = __shfl_xor_sync(0xffffffffu, r, m);
    r = MAX ? fmaxf(r, got) : r + got;
  }
  return r;
}

// 8 or 16 bytes at logical byte `off` of row `row` of a 128-byte-swizzled
// region (16-byte chunk c of row r sits at chunk c ^ (r % 8)).
__device__ __forceinline__ void st_sw128_u2(uint8_t* base, int row, int off, uint32_t a, uint32_t b) {
  *reinterpret_cast<uint2*>(base + row * 128 + ((((off >> 4) ^ (row & 7)) << 4) | (off & 15))) = make_uint2(a, b);
}
__device__ __forceinline__ void st_sw128_u4(uint8_t* base, int row, int off, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d) {
  *reinterpret_cast<uint4*>(base + row * 128 + (((off >> 4) ^ (row & 7)) << 4)) = make_uint4(a, b, c, d);
}

template <bool FP8, int NR>
__global__ void __launch_bounds__(pm_threads(FP8, NR), 1)
    attn_pm_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ AttnParams p) {
  constexpr int D = 128;
  constexpr int H = 8;                  // columns of one softmax thread
  constexpr int LH = 3;
  constexpr int CG = NR / H;            // column groups
  constexpr int SMW = 4 * CG;           // softmax warps
  constexpr int WK = SMW, WU = SMW + 1, WV = SMW + 2, WQ = SMW + 3;  // other roles
  constexpr int KV = FP8 ? kGroups * kBox : kGroups * 2 * kBox;
  // FP8: the hi and lo E4M3 terms of Q (and of P) are the two halves of N, so
  // one instruction covers both; the softmax and the epilogue add the halves
  constexpr int SW = FP8 ? 2 * NR : NR;  // UMMA N = TMEM columns of S^T and of O^T
  constexpr uint32_t IDESC_QK = FP8 ? umma_idesc_e4m3(128, SW) : umma_idesc_bf16(128, SW);
  constexpr uint32_t IDESC_PV = IDESC_QK | (1u << 15) | (1u << 16);  // A (V^T) and B (P^T) MN-major
  // pages go through in pairs: S^T buffer / P^T buffer 2 s + e holds page e of
  // the pair in slot s (two slots); O^T after the four S^T buffers
  constexpr uint32_t TM_O = 4 * SW;
  constexpr uint32_t TMEM_COLS = 5 * SW <= 128 ? 128 : (5 * SW <= 256 ? 256 : 512);
  constexpr int BPR = 64 / NR;      // P^T buffers per 128-byte row (2 NR bytes each)
  static_assert(NR == 16 || NR == 32, "row tiles of 16 or 32");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int NK = p.nstages, NV = p.nv, NQ = p.nq, QBUF = p.qbuf;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* kempty = kfull + NK;   // QK finished reading the K stage
  uint64_t* vfull = kempty + NK;
  uint64_t* vempty = vfull + NV;   // PV finished reading the V stage
  uint64_t* sfull = vempty + NV;   // [2 pair slots] S^T of the pair written
  uint64_t* pfull = sfull + 2;     // [2] P^T of the pair written (the softmax warps)
  uint64_t* pvdone = pfull + 2;    // [2] PV of the pair retired
  uint64_t* qfull = pvdone + 2;    // [2] bf16 Q tile landed
  uint64_t* qempty = qfull + 2;    // [2] last QK of the sequence retired
  uint64_t* qcv = qempty + 2;      // [2] FP8: E4M3 Q terms and row scales written
  uint64_t* qsfree = qcv + 2;      // [2] FP8: the softmax warps have read the row scales
  uint64_t* mdone = qsfree + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mdone + 1);
  int* abortf = reinterpret_cast<int*>(mdone + 2);  // the CTA's give-up flag
  const Waits wt{p.err, abortf, p.wait_ns};
  int32_t* scan = reinterpret_cast<int32_t*>(smem + p.off_scan);
  // [2 pages][4 quadrants][NR] column maxima, [4][NR] column sums, [2][NR] Q row scales
  float* cmax = reinterpret_cast<float*>(smem + p.off_ml);
  float* lsm = cmax + 8 * NR;
  float* qsc = lsm + 4 * NR;
  int* pvote = reinterpret_cast<int*>(qsc + 2 * NR);  // [2 pages][CG column groups]
  const bool sparse = p.sparse != 0;
  const int Hk = p.num_kv_heads, T = p.qo_len, G = p.group;
  const int nitems = sparse ? p.batch * Hk : p.batch;
  int32_t* warp_tot = scan + nitems + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NK; ++i) { mbar_init(&kfull[i], 1); mbar_init(&kempty[i], 1); }
    for (int i = 0; i < NV; ++i) { mbar_init(&vfull[i], 1); mbar_init(&vempty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], SMW);
      mbar_init(&pvdone[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
      mbar_init(&qcv[i], 1);
      mbar_init(&qsfree[i], SMW);
    }
    mbar_init(mdone, 1);
    *abortf = 0;
    for (int i = 0; i < 2 * CG; ++i) pvote[i] = -1;
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

  if (warp == WU) {
    tmem_alloc(tslot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  uint8_t* qbase = smem + p.off_q;
  uint8_t* qf8 = smem + p.off_qf8;  // FP8: [2 sequences][2 terms][NR rows][128 B]
  uint8_t* preg = smem + p.off_p;
  uint8_t* kring = smem + p.off_stage;
  uint8_t* vring = smem + p.off_vring;

  if (warp == WK || warp == WV) {
    // ------------------------------------------- TMA producers: K (+Q) and V
    if (lane == 0) {
      const bool is_v = warp == WV;
      prefetch_tensormap(&kv_map);
      if (!is_v) prefetch_tensormap(&q_map);
      const uint64_t pol = policy_evict_first();
      const int sub_rows = Hk * kSub;
      const uint32_t qbytes = static_cast<uint32_t>(2 * 64 * 2 * G * T);
      const int n = is_v ? NV : NK;
      uint64_t* fullb = is_v ? vfull : kfull;
      uint64_t* emptyb = is_v ? vempty : kempty;
      uint8_t* ring = is_v ? vring : kring;
      int it = 0, sq = 0, st = 0;
      uint32_t eph = 1;  // parity of the empty barrier phase that frees stage st
      bool alive = true;
      for (SeqCursor cur = cursor_first(scan, nitems, Hk, sparse, u0);
           alive && (sparse ? cur.s : cur.b) < nitems && seq_in_range(cur, u1, p.setup);
           cursor_next(cur, scan, nitems, Hk, sparse), ++sq) {
        if (!is_v) {
          // the bf16 tile is free once the UMMAs (bf16) or the quantiser (FP8)
          // of the sequence NQ back are done with it
          const int qb = sq % NQ;
          if (sq >= NQ && !mbar_wait(FP8 ? &qcv[qb] : &qempty[qb], static_cast<uint32_t>(sq / NQ - 1) & 1u, wt)) {
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
        }
        const int64_t j0 = seq_j0(cur, u0, p.setup), j1 = seq_j1(cur, u1, p.setup);
        const int L = p.sub_k != nullptr ? p.kv_lens[cur.b] : 0;  // P32 tables: used entries
        for (int64_t j = j0; j < j1; ++j, ++it) {
          if (!is_v && p.withhold >= 0 && it >= p.withhold) {  // tests of the give-up path only
            alive = false;
            break;
          }
          const int blk = sparse ? p.plan_blocks[static_cast<int64_t>(cur.s) * p.plan_cap + j]
                                 : static_cast<int>(j);
          const int64_t row = static_cast<int64_t>(cur.b) * p.max_pages + blk;
          int slot = 0;
          if (p.sub_k == nullptr) {
            slot = p.page_table[row];
            if (slot < 0 || slot >= p.num_slots) {
              if (!is_v) atomicOr(p.err, TRTV_DEVERR_PAGE_ID);
              slot = 0;
            }
          }
          const int64_t buf = static_cast<int64_t>(slot) * p.slot_stride + (is_v ? 1 : 0);
          if (it >= n && !mbar_wait(&emptyb[st], eph, wt)) {
            alive = false;
            break;
          }
          uint8_t* dst = ring + st * KV;
          mbar_arrive_expect_tx(&fullb[st], KV);
#pragma unroll
          for (int hb = 0; hb < (FP8 ? 1 : 2); ++hb)
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
              const int sp = p.sub_k != nullptr
                                 ? p32_entry(is_v ? p.sub_v : p.sub_k, row * kGroups + g,
                                             blk * kGroups + g, L, p.num_subpages, p.err)
                                 : static_cast<int>(buf * kGroups + g);
              tma_load_2d(dst + (hb * kGroups + g) * kBox, &kv_map, &fullb[st], hb * 64,
                          sp * sub_rows + cur.h * kSub, pol);
            }
          if (++st == n) {
            st = 0;
            eph ^= 1u;
          }
        }
      }
      // never leave copies in flight
      for (int k = (it > n ? it - n : 0); k < it; ++k)
        mbar_drain(&fullb[k % n], static_cast<uint32_t>(k / n) & 1u, wt);
      if (!is_v && sq >= 1)
        mbar_drain(&qfull[(sq - 1) % NQ], static_cast<uint32_t>((sq - 1) / NQ) & 1u, wt);
    }
  } else if (warp == WU) {
    // ----------------------------------------------------------- UMMA issuer
    // The whole warp runs the loop (uniform control flow, operands in uniform
    // registers) and one elected lane issues; lane 0 waits for the barriers.
    // Descriptors are built once and moved by byte offsets; ring positions
    // advance by increments (no division in the loop).
    const uint64_t kd0 = umma_desc_sw128(smem_u32(kring));
    const uint64_t qd0 = umma_desc_sw128(smem_u32(FP8 ? qf8 : qbase));
    const uint64_t vd0 = FP8 ? umma_desc_sw128_lbo_sbo(smem_u32(vring), 1024, 1024)
                             : umma_desc_sw128_mn(smem_u32(vring), KV / 2);
    const uint64_t pd0 = FP8 ? umma_desc_sw128_lbo_sbo(smem_u32(preg), 1024, 1024)
                             : umma_desc_sw128_mn(smem_u32(preg), kPmPRegion);
    const uint32_t qhalf = static_cast<uint32_t>(QBUF / 2);
    auto wait1 = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, lane != 0 || mbar_wait(bar, par, wt));
    };
    bool alive = true;
    int ks = 0, vs = 0;
    uint32_t kph = 0, vph = 0;
    uint32_t qps = 0;             // pair slot of the next QK pair
    uint32_t vps = 0, vpph = 0;   // pair slot of the next PV pair, and its pfull phase
    // PV of a pair: n pages; `first`: the sequence's first pair (O^T starts over)
    auto issue_pv = [&](int n, bool first) {
      if (!alive) return;
      if (!wait1(&pfull[vps], vpph)) {
        alive = false;
        return;
      }
      for (int e = 0; e < n; ++e) {
        if (!wait1(&vfull[vs], vph)) {
          alive = false;
          return;
        }
        tc_fence_after();
        const uint64_t va = desc_add(vd0, static_cast<uint32_t>(vs * KV));
        const int bi = 2 * vps + e;
        const uint64_t pbd = desc_add(pd0, static_cast<uint32_t>((bi / BPR) * kPmPRegion + (bi % BPR) * 2 * NR));
        const bool zero = first && e == 0;
        // FP8: 32 positions per UMMA (32 V rows of 128 B = 4 KB), the 128 head
        // dims one swizzle atom, N = both P terms.  bf16: 16 positions per
        // UMMA, the head dims' two 64-column atoms of the V stage KV / 2 apart.
        constexpr uint32_t PSTEP = FP8 ? 4096 : 2048;
#pragma unroll
        for (int h4 = 0; h4 < (FP8 ? 1 : 2); ++h4) {
          uint64_t a[4], b[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a[i] = desc_add(va, (4 * h4 + i) * PSTEP);
            b[i] = desc_add(pbd, (4 * h4 + i) * PSTEP);
          }
          umma4_elect<FP8>(tmem + TM_O, a, b, IDESC_PV, (!zero || h4 > 0) ? 1u : 0u);
        }
        umma_commit_elect(&vempty[vs]);
        if (++vs == NV) {
          vs = 0;
          vph ^= 1u;
        }
      }
      umma_commit_elect(&pvdone[vps]);
      vps ^= 1u;
      if (vps == 0) vpph ^= 1u;
    };
    int sq = 0, pend_n = 0;
    bool pend_first = false;
    for (SeqCursor cur = cursor_first(scan, nitems, Hk, sparse, u0);
         alive && (sparse ? cur.s : cur.b) < nitems && seq_in_range(cur, u1, p.setup);
         cursor_next(cur, scan, nitems, Hk, sparse), ++sq) {
      const int qb = sq % NQ, qs = sq & 1;
      if (!wait1(FP8 ? &qcv[qs] : &qfull[qb], static_cast<uint32_t>(FP8 ? sq >> 1 : sq / NQ) & 1u)) {
        alive = false;
        break;
      }
      const uint64_t qd = desc_add(qd0, static_cast<uint32_t>(FP8 ? qs * 2 * NR * 128 : qb * QBUF));
      const int64_t j0 = seq_j0(cur, u0, p.setup), j1 = seq_j1(cur, u1, p.setup);
      for (int64_t j = j0; j < j1 && alive; j += 2) {
        // S^T buffers of slot qps were last read by the softmax of the pair two
        // back, whose P this warp has already waited for (that PV went first)
        const int n = j + 1 < j1 ? 2 : 1;
        for (int e = 0; e < n; ++e) {
          if (!wait1(&kfull[ks], kph)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint64_t ka = desc_add(kd0, static_cast<uint32_t>(ks * KV));
          const uint32_t sd = tmem + (2 * qps + e) * SW;
          // FP8: K = 32 head dims per UMMA, N = the hi and lo terms of the rows;
          // bf16: K = 16, the head dims' two 64-column halves KV / 2 (K page)
          // and qhalf (Q tile) apart
#pragma unroll
          for (int h4 = 0; h4 < (FP8 ? 1 : 2); ++h4) {
            uint64_t a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              a[i] = desc_add(ka, FP8 ? i * 32 : h4 * (KV / 2) + i * 32);
              b[i] = desc_add(qd, FP8 ? i * 32 : h4 * qhalf + i * 32);
            }
            umma4_elect<FP8>(sd, a, b, IDESC_QK, h4 > 0 ? 1u : 0u);
          }
          umma_commit_elect(&kempty[ks]);
          if (++ks == NK) {
            ks = 0;
            kph ^= 1u;
          }
        }
        if (!alive) break;
        umma_commit_elect(&sfull[qps]);
        if (j + n == j1) umma_commit_elect(FP8 ? &qempty[qs] : &qempty[qb]);
        qps ^= 1u;
        if (pend_n > 0) issue_pv(pend_n, pend_first);
        pend_n = n;
        pend_first = j == j0;
      }
      // the sequence's last PV goes out now: its epilogue must not wait for
      // the next sequence's Q tile and first QK
      if (pend_n > 0) issue_pv(pend_n, pend_first);
      pend_n = 0;
    }
    umma_commit_elect(mdone);
    if (lane == 0) mbar_drain(mdone, 0, wt);
    __syncwarp();
  } else if (FP8 && warp == WQ) {
    // ------------------------------------------------ FP8: Q quantiser warp
    // Each sequence's bf16 Q tile -> two E4M3 terms (hi = E4M3(x), lo =
    // E4M3(x - hi)) of q / 2^e with a power-of-two scale per row; the E4M3
    // tiles and row scales are double-buffered by sequence parity.
    bool dead = false;
    int sq = 0;
    const int rows = G * T;
    for (SeqCursor cur = cursor_first(scan, nitems, Hk, sparse, u0);
         (sparse ? cur.s : cur.b) < nitems && seq_in_range(cur, u1, p.setup);
         cursor_next(cur, scan, nitems, Hk, sparse), ++sq) {
      const int qb = sq % NQ, qs = sq & 1;
      if (!dead)
        dead = __any_sync(0xffffffffu, !mbar_wait(&qfull[qb], static_cast<uint32_t>(sq / NQ) & 1u, wt));
      if (!dead && sq >= 2)
        dead = __any_sync(0xffffffffu, !mbar_wait(&qempty[qs], static_cast<uint32_t>((sq >> 1) - 1) & 1u, wt));
      if (!dead && sq >= 2)
        dead = __any_sync(0xffffffffu, !mbar_wait(&qsfree[qs], static_cast<uint32_t>((sq >> 1) - 1) & 1u, wt));
      uint8_t* qhi = qf8 + qs * 2 * NR * 128;
      for (int r = lane; r < rows; r += 32)
        qsc[qs * NR + r] = quantize_q_row(qbase + qb * QBUF, QBUF / 2, qhi, qhi + NR * 128, r);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qcv[qs]);
    }
  } else if (warp < SMW) {
    // -------------------------------------------------- softmax and epilogue
    const int q = warp & 3;          // TMEM lane quadrant: positions 32 q .. 32 q + 31
    const int cg = warp >> 2;        // column group
    const int col0 = cg * H;
    const int kpos = 32 * q + lane;  // position in the page; head dim in the epilogue
    const int rows = G * T, lg = p.lg_group;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
    bool dead = false;
    int it = 0, ip = 0, sq = 0;  // pages, pairs and sequences so far
    int Lc = p.kv_lens[cursor_first(scan, nitems, Hk, sparse, u0).b];  // kv_len of the sequence about to start
    for (SeqCursor cur = cursor_first(scan, nitems, Hk, sparse, u0);
         (sparse ? cur.s : cur.b) < nitems && seq_in_range(cur, u1, p.setup);
         cursor_next(cur, scan, nitems, Hk, sparse), ++sq) {
      const int L = Lc;
      {  // the next sequence's kv_len loads a whole sequence ahead of its use
        SeqCursor nx = cur;
        cursor_next(nx, scan, nitems, Hk, sparse);
        if ((sparse ? nx.s : nx.b) < nitems) Lc = p.kv_lens[nx.b];
      }
      const int64_t j0 = seq_j0(cur, u0, p.setup), j1 = seq_j1(cur, u1, p.setup);
      // logit scale per column in the log2 domain (FP8: times the row's Q scale)
      float sc[H];
#pragma unroll
      for (int i = 0; i < H; ++i) sc[i] = p.scale_log2;
      if constexpr (FP8) {
        const int qs = sq & 1;
        if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(&qcv[qs], static_cast<uint32_t>(sq >> 1) & 1u, wt));
#pragma unroll
        for (int i = 0; i < H; ++i) sc[i] *= col0 + i < rows ? qsc[qs * NR + col0 + i] : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&qsfree[qs]);
      }
      // mth: the column's reference maximum + 8 (-inf until a first value)
      float mth[H], ls[H];
#pragma unroll
      for (int i = 0; i < H; ++i) {
        mth[i] = -INFINITY;
        ls[i] = 0.f;
      }
      for (int64_t j = j0; j < j1; j += 2, ++ip) {
        const int n = j + 1 < j1 ? 2 : 1;     // pages of this pair
        const int ps = ip & 1;                 // pair slot
        const uint32_t pph = static_cast<uint32_t>(ip >> 1) & 1u;
        int blk[2], pos0[2];
        uint32_t tokmask[2] = {0xffffffffu, 0xffffffffu};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          blk[e] = static_cast<int>(j) + e;
          if (sparse && e < n) {
            blk[e] = p.plan_blocks[static_cast<int64_t>(cur.s) * p.plan_cap + j + e];
            tokmask[e] = p.plan_masks[static_cast<int64_t>(cur.s) * p.plan_cap + j + e];
          }
          pos0[e] = blk[e] * kPage;
        }
        if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(&sfull[ps], pph, wt));
        tc_fence_after();
        float x[2][H];
        bool over = false;  // a value above its column's reference maximum + 8
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (e >= n) {
#pragma unroll
            for (int i = 0; i < H; ++i) x[e][i] = -INFINITY;
            continue;
          }
          const uint32_t sa = tl + (2 * ps + e) * SW + col0;
          uint32_t r[H];
          tmem_ld_async(sa, r);
          if constexpr (FP8) {  // S = (Q_hi + Q_lo) K^T: add the lo half of N
            uint32_t r2[H];
            tmem_ld_async(sa + NR, r2);
            tmem_ld_wait_dep(r);
            tmem_ld_wait_dep(r2);
#pragma unroll
            for (int i = 0; i < H; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
          } else {
            tmem_ld_wait_dep(r);
          }
          const int pos = pos0[e] + kpos;
          const bool masked = sparse || rows < NR || pos0[e] + kPage - 1 > L - T;
#pragma unroll
          for (int i = 0; i < H; ++i) {
            float v = __uint_as_float(r[i]) * sc[i];
            if (masked) {
              const int c = col0 + i, t = c >> lg;
              const bool ok = c < rows && pos <= L - T + t && ((tokmask[e] >> t) & 1u);
              v = ok ? v : -INFINITY;
            }
            x[e][i] = v;
            over |= v > mth[i];
          }
        }
        // The reference maxima move only when some value of the pair exceeds
        // them by more than 8 (log2 domain): the warps of the column group
        // vote, and only then are the exact column maxima exchanged (always on
        // a sequence's first pair, where the references are -inf).  The vote
        // slot holds the pair index of its last "yes", double-buffered by pair
        // parity; every warp of the group reads the same slot, so the barriers
        // below are taken alike.
        volatile int* vote = pvote + (ip & 1) * CG + cg;
        if (__any_sync(0xffffffffu, over) && lane == 0) *vote = ip;
        named_barrier(2 + cg, 128);
        if (*vote == ip) {
          float red[H];
#pragma unroll
          for (int i = 0; i < H; ++i) red[i] = fmaxf(x[0][i], x[1][i]);
          const float cm = lane_col_reduce<H, true>(red, lane);
          float* cb = cmax + (ip & 1) * 4 * NR;
          if ((lane & ((1 << (5 - LH)) - 1)) == 0) cb[q * NR + col0 + (lane >> (5 - LH))] = cm;
          named_barrier(2 + cg, 128);
          float mp[H];
#pragma unroll
          for (int i = 0; i < H; i += 4) {
            float4 a = *reinterpret_cast<const float4*>(cb + col0 + i);
#pragma unroll
            for (int qq = 1; qq < 4; ++qq) {
              const float4 b = *reinterpret_cast<const float4*>(cb + qq * NR + col0 + i);
              a.x = fmaxf(a.x, b.x); a.y = fmaxf(a.y, b.y); a.z = fmaxf(a.z, b.z); a.w = fmaxf(a.w, b.w);
            }
            mp[i] = a.x; mp[i + 1] = a.y; mp[i + 2] = a.z; mp[i + 3] = a.w;
          }
          // first values of a column set its reference; a rise by more than 8
          // rescales the column's O^T and sum (the same decision in every
          // thread of the group: it depends on shared values only)
          bool need = false;
#pragma unroll
          for (int i = 0; i < H; ++i) {
            if (mth[i] == -INFINITY) mth[i] = mp[i] + kRescaleLog2;
            else need |= mp[i] > mth[i];
          }
          if (need) {
            // O^T must be stable: PV of the previous pair (of this sequence:
            // a reference was set on an earlier pair) has retired
            const int pv = ip - 1;
            if (!dead)
              dead = __any_sync(0xffffffffu, !mbar_wait(&pvdone[pv & 1], static_cast<uint32_t>(pv >> 1) & 1u, wt));
            tc_fence_after();
            float alpha[H];
#pragma unroll
            for (int i = 0; i < H; ++i) {
              const bool ni = mp[i] > mth[i];
              alpha[i] = ni ? fast_exp2(mth[i] - mp[i] - kRescaleLog2) : 1.f;
              ls[i] *= alpha[i];
              if (ni) mth[i] = mp[i] + kRescaleLog2;
            }
#pragma unroll
            for (int half = 0; half < (FP8 ? 2 : 1); ++half) {  // FP8: the P_hi and P_lo parts of O^T
              uint32_t o[H];
              tmem_ld_async(tl + TM_O + half * NR + col0, o);
              tmem_ld_wait_dep(o);
#pragma unroll
              for (int i = 0; i < H; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha[i]);
              tmem_st8(tl + TM_O + half * NR + col0, o);
            }
            tmem_st_wait();
          }
        }
        // P^T of the pair into buffers 2 ps, 2 ps + 1, once PV of the pair two
        // back (the same slot) has read them
        if (ip >= 2 && !dead)
          dead = __any_sync(0xffffffffu, !mbar_wait(&pvdone[ps], static_cast<uint32_t>((ip >> 1) - 1) & 1u, wt));
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (e >= n) continue;
          float pv[H];
#pragma unroll
          for (int i = 0; i < H; ++i) {
            pv[i] = mth[i] == -INFINITY ? 0.f : fast_exp2(x[e][i] - mth[i] + kRescaleLog2);
            ls[i] += pv[i];
          }
          const int bi = 2 * ps + e;
          uint8_t* pr = preg + (bi / BPR) * kPmPRegion;
          const int pbyte = (bi % BPR) * 2 * NR;
          if constexpr (FP8) {
            uint32_t wh[H / 4], wl[H / 4];
#pragma unroll
            for (int i = 0; i < H / 4; ++i) {
              uint32_t h0, l0, h1, l1;
              split_e4m3x2(__floats2half2_rn(pv[4 * i], pv[4 * i + 1]), h0, l0);
              split_e4m3x2(__floats2half2_rn(pv[4 * i + 2], pv[4 * i + 3]), h1, l1);
              wh[i] = (h0 & 0xFFFFu) | (h1 << 16);
              wl[i] = (l0 & 0xFFFFu) | (l1 << 16);
            }
            st_sw128_u2(pr, kpos, pbyte + col0, wh[0], wh[1]);
            st_sw128_u2(pr, kpos, pbyte + NR + col0, wl[0], wl[1]);
          } else {
            uint32_t w[H / 2];
#pragma unroll
            for (int i = 0; i < H / 2; ++i) {
              __nv_bfloat162 pk = __floats2bfloat162_rn(pv[2 * i], pv[2 * i + 1]);
              w[i] = *reinterpret_cast<uint32_t*>(&pk);
            }
            st_sw128_u4(pr, kpos, pbyte + 2 * col0, w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        // V rows at or past kv_len may hold anything (NaN included): P is zero
        // there, but 0 * NaN is not, so warp 0 zeroes them before PV reads V.
        if (warp == 0) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int nvalid = L - pos0[e];
            if (e >= n || nvalid >= kPage) continue;
            const int vs = (it + e) % NV;
            if (!dead)
              dead = __any_sync(0xffffffffu, !mbar_wait(&vfull[vs], static_cast<uint32_t>((it + e) / NV) & 1u, wt));
            uint8_t* vst = vring + vs * KV;
            constexpr int NHALF = FP8 ? 1 : 2;  // 128-byte column blocks per token row
            const int nchunks = (kPage - nvalid) * 8 * NHALF;
            for (int idx = lane; idx < nchunks; idx += 32) {
              const int tok = nvalid + idx / (8 * NHALF), part = idx % (8 * NHALF);
              *reinterpret_cast<uint4*>(vst + ((part >> 3) * kGroups + tok / kSub) * kBox + (tok % kSub) * 128 +
                                        (part & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[ps]);
        it += n;
      }
      // ------------------------------------------------------- sequence end
      const int last = ip - 1;
      if (!dead)
        dead = __any_sync(0xffffffffu, !mbar_wait(&pvdone[last & 1], static_cast<uint32_t>(last >> 1) & 1u, wt));
      tc_fence_after();
      const float cs = lane_col_reduce<H, false>(ls, lane);
      if ((lane & ((1 << (5 - LH)) - 1)) == 0) lsm[q * NR + col0 + (lane >> (5 - LH))] = cs;
      named_barrier(2 + cg, 128);
      float lt[H];
#pragma unroll
      for (int i = 0; i < H; i += 4) {
        float4 a = *reinterpret_cast<const float4*>(lsm + col0 + i);
#pragma unroll
        for (int qq = 1; qq < 4; ++qq) {
          const float4 b = *reinterpret_cast<const float4*>(lsm + qq * NR + col0 + i);
          a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
        }
        lt[i] = a.x; lt[i + 1] = a.y; lt[i + 2] = a.z; lt[i + 3] = a.w;
      }
      uint32_t o[H];
      tmem_ld_async(tl + TM_O + col0, o);
      if constexpr (FP8) {  // O^T = V^T P_hi^T + V^T P_lo^T
        uint32_t o2[H];
        tmem_ld_async(tl + TM_O + NR + col0, o2);
        tmem_ld_wait_dep(o);
        tmem_ld_wait_dep(o2);
#pragma unroll
        for (int i = 0; i < H; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) + __uint_as_float(o2[i]));
      } else {
        tmem_ld_wait_dep(o);
      }
      const bool whole = seq_whole(cur, u0, u1, p.setup);
      const int64_t slot = seq_slot(cur, u0, p.setup);
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const int c = col0 + i;
        if (c >= rows) continue;
        const float inv = lt[i] > 0.f ? 1.f / lt[i] : 0.f;
        const float val = __uint_as_float(o[i]) * inv;
        if (whole) {
          const int t = c >> lg, g = c & (G - 1);
          const int64_t orow = ((static_cast<int64_t>(cur.b) * T + t) * p.num_q_heads +
                                static_cast<int64_t>(cur.h) * G + g) * D + kpos;
          if (p.out_f32) static_cast<float*>(p.out)[orow] = val * p.v_scale;
          else static_cast<__nv_bfloat16*>(p.out)[orow] = __float2bfloat16(val * p.v_scale);
        } else {
          p.ws_o[(slot * p.rows_pad + c) * D + kpos] = val;
          if (kpos == 0)
            p.ws_lse[slot * p.rows_pad + c] = lt[i] > 0.f ? mth[i] - kRescaleLog2 + __log2f(lt[i]) : -INFINITY;
        }
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WU) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace trtv
