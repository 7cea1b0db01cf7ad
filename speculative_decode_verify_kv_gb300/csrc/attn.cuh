// attn.cuh -- split-KV ladder verify attention over P128 pages read as
// grouped-HND [4][kv_head][32][head_dim] sub-pages (dense and MSA sparse).
//
// Sources: "Eagle3 for M3 MSA path + CUDA graphs compatibility" (fork PR #3),
// commit "... verify" (ladder: token t attends kv_len - qo_len + t + 1
// positions; sparse GQA over selected blocks); "Default Minimax-m3 to unified
// draft-target kv manager" (#17835), "Grouped-HND draft KV transfer" (page
// layout); "wrap up eagle changes in m3 side branch" (#18066), view commit
// (K page at slot * stride, V page at slot * stride + 1).
//
// One CTA per SM ("stream-K" split): the work units are the pages (dense) or
// the unique selected blocks (sparse) of every (request, KV head) sequence,
// concatenated in sequence order; CTA c takes units [c W / P, (c+1) W / P).
// A sequence that one CTA covers whole is written as final output; the
// pieces of a cut sequence are written as (normalised output, log2-sum-exp)
// partials, which the split-combine kernel (combine_kernel) merges right
// after, on every SM at once.
//
// Roles: warp 8 issues TMA tiled loads of each page's K and V sub-pages
// (128B swizzle) into an NST-stage ring guarded by full/empty mbarriers.
// Warps 0..7 compute: warp w owns row tile w % MT (16 rows of the
// (token, group head) tile, row = t * group_pad + g) and the token slice
// (w / MT) * 16 MT .. + 16 MT of every page.  QK^T and PV run on mma.sync
// m16n8k16 (bf16, or f16 when the cache is FP8), fp32 accumulation, online
// softmax in the log2 domain.  At the end of a sequence the 8 / MT slice
// partials of each row tile are merged in fixed order through shared memory.
#pragma once

#include "common.cuh"

namespace trtv {

template <int D>
struct Shape {
  static constexpr int KS = D / 16;  // k-steps of QK^T
  static constexpr int DT = D / 8;   // n-tiles (8 columns) of PV
};

// Loads the A fragments of Q for one 16-row tile.  Rows beyond the
// (qo_len x group) tile are zero.  FP8 caches use f16 operands and a
// permuted k order (k-step ks, lane quad c: head dims 32c + 4ks + {0..3}).
template <bool FP8, int D>
__device__ __forceinline__ void load_q_frags(const __nv_bfloat16* q, int T, int Hq, int G, int Gp,
                                             int b, int h, int mt, uint32_t (&qa)[D / 16][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const __nv_bfloat16* rowp[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int r = mt * 16 + g + 8 * hh;
    const int t = r / Gp, gl = r % Gp;
    rowp[hh] = (t < T && gl < G)
                   ? q + ((static_cast<int64_t>(b) * T + t) * Hq + static_cast<int64_t>(h) * G + gl) * D
                   : nullptr;
  }
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t lo = 0, hi = 0;
      if (rowp[hh] != nullptr) {
        if constexpr (FP8) {
          const uint2 v = __ldg(reinterpret_cast<const uint2*>(rowp[hh] + 32 * c + 4 * ks));
          lo = bf16x2_to_f16x2(v.x);
          hi = bf16x2_to_f16x2(v.y);
        } else {
          lo = __ldg(reinterpret_cast<const uint32_t*>(rowp[hh] + 16 * ks + 2 * c));
          hi = __ldg(reinterpret_cast<const uint32_t*>(rowp[hh] + 16 * ks + 8 + 2 * c));
        }
      }
      qa[ks][hh] = lo;       // a0 (row g) / a1 (row g+8): k = 2c, 2c+1
      qa[ks][2 + hh] = hi;   // a2 / a3: k = 2c+8, 2c+9
    }
  }
}

// Sequence cursor over the CTA's unit range.  Dense: items are requests
// (every KV head of a request has the same page count); sparse: items are
// (request, KV head) sequences.
struct SeqCursor {
  int b, h, s;
  int64_t start, units;
};

__device__ __forceinline__ int64_t item_start(const int32_t* scan, int i, int Hk, bool sparse) {
  return sparse ? static_cast<int64_t>(scan[i]) : static_cast<int64_t>(scan[i]) * Hk;
}

__device__ __forceinline__ void cursor_fill(SeqCursor& cur, const int32_t* scan, int Hk,
                                            bool sparse) {
  if (sparse) {
    cur.start = scan[cur.s];
    cur.units = scan[cur.s + 1] - scan[cur.s];
  } else {
    const int64_t u = scan[cur.b + 1] - scan[cur.b];
    cur.start = static_cast<int64_t>(scan[cur.b]) * Hk + cur.h * u;
    cur.units = u;
  }
}

// First sequence holding unit u0 (u0 < W).
__device__ __forceinline__ SeqCursor cursor_first(const int32_t* scan, int n, int Hk, bool sparse,
                                                  int64_t u0) {
  int lo = 0, hi = n;  // last item i with start(i) <= u0
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (item_start(scan, mid, Hk, sparse) <= u0) lo = mid; else hi = mid - 1;
  }
  SeqCursor cur;
  if (sparse) {
    cur.s = lo; cur.b = lo / Hk; cur.h = lo % Hk;
  } else {
    const int64_t u = scan[lo + 1] - scan[lo];
    cur.b = lo;
    cur.h = static_cast<int>((u0 - static_cast<int64_t>(scan[lo]) * Hk) / u);
    cur.s = lo * Hk + cur.h;
  }
  cursor_fill(cur, scan, Hk, sparse);
  return cur;
}

__device__ __forceinline__ void cursor_next(SeqCursor& cur, const int32_t* scan, int n, int Hk,
                                            bool sparse) {
  if (sparse) {
    do { ++cur.s; } while (cur.s < n && scan[cur.s + 1] == scan[cur.s]);
    cur.b = cur.s / Hk; cur.h = cur.s % Hk;
  } else {
    if (++cur.h == Hk) {
      cur.h = 0;
      do { ++cur.b; } while (cur.b < n && scan[cur.b + 1] == scan[cur.b]);
    }
    cur.s = cur.b * Hk + cur.h;
  }
  if ((sparse ? cur.s : cur.b) < n) cursor_fill(cur, scan, Hk, sparse);
}

// Stream-K with a setup charge: every non-empty sequence owns `setup` virtual
// units ahead of its pages (or blocks), standing for the fixed cost of
// starting it (epilogue of the previous one, Q, pipeline refill), so a CTA
// that starts more sequences gets fewer pages.  A sequence spans virtual
// units [start, start + units); its real units begin at rs = start + setup.
__device__ __forceinline__ bool seq_in_range(const SeqCursor& c, int64_t u1, int setup) {
  return c.start + setup < u1;
}
// real units [j0, j1) of the sequence inside the CTA's range [u0, u1)
__device__ __forceinline__ int64_t seq_j0(const SeqCursor& c, int64_t u0, int setup) {
  const int64_t rs = c.start + setup;
  return (u0 > rs ? u0 : rs) - rs;
}
__device__ __forceinline__ int64_t seq_j1(const SeqCursor& c, int64_t u1, int setup) {
  const int64_t e = c.start + c.units;
  return (u1 < e ? u1 : e) - (c.start + setup);
}
// no other CTA holds a real unit of the sequence
__device__ __forceinline__ bool seq_whole(const SeqCursor& c, int64_t u0, int64_t u1, int setup) {
  return u0 <= c.start + setup && c.start + c.units <= u1;
}
// workspace slot of a cut piece: 2c for the piece that began before the CTA's
// range (at most one), 2c + 1 for the one that runs past it (at most one)
__device__ __forceinline__ int64_t seq_slot(const SeqCursor& c, int64_t u0, int setup) {
  return 2 * static_cast<int64_t>(blockIdx.x) + (c.start + setup <= u0 ? 0 : 1);
}

// Virtual units of item i (a request's per-KV-head page count, or a sparse
// sequence's block count) plus the setup charge; 0 for an empty item.
__device__ __forceinline__ int32_t seq_units(const AttnParams& p, int i, int T, bool sparse) {
  int32_t u;
  if (sparse) {
    u = p.plan_count[i];
  } else {
    const int L = p.kv_lens[i];
    if (len_valid(L, T, p.max_pages)) {
      u = (L + kPage - 1) / kPage;
    } else {
      if (blockIdx.x == 0) atomicOr(p.err, TRTV_DEVERR_KV_LEN);
      u = 0;
    }
  }
  return u > 0 ? u + p.setup : 0;
}

// Stream-K bookkeeping for the split-combine kernel.  CTA k (k >= 1) starts at
// unit B_k = begin(k).  If B_k falls strictly inside the real units of a
// sequence whose real units began in CTA k - 1's range (B_{k-1} <= rs < B_k),
// boundary k is the first one that cuts it: CTA k records the sequence and its
// contributors c_first = k - 1 .. cta_of_unit(start + units - 1).  Every boundary is recorded (b = -1 when it
// starts no cut), so each cut sequence is described exactly once per call.
// Called by one thread of every CTA, before any early exit.
__device__ __forceinline__ void write_split_desc(const AttnParams& p, const int32_t* scan, int n, int Hk,
                                                 bool sparse, int64_t W) {
  const int64_t k = blockIdx.x, P = p.num_ctas;
  if (k == 0 || k >= P) return;
  SplitDesc d;
  d.b = -1; d.h = 0; d.c_first = 0; d.nc = 0; d.first_off = 0; d.pad = 0;
  d.W = W;
  const int64_t B = cta_unit_begin(k, W, P);
  if (B < W) {
    const SeqCursor cur = cursor_first(scan, n, Hk, sparse, B);
    const int64_t Bp = cta_unit_begin(k - 1, W, P);
    const int64_t rs = cur.start + p.setup;  // first real unit
    if (rs < B && rs >= Bp) {
      d.b = cur.b;
      d.h = cur.h;
      d.c_first = static_cast<int>(k - 1);
      d.nc = static_cast<int>(cta_of_unit(cur.start + cur.units - 1, W, P) - (k - 1) + 1);
      d.first_off = Bp < rs ? 1 : 0;
    }
  }
  p.splits[k] = d;
}

// Sub-page buffer indices (units of one [Hk, 32, D] sub-page of the pool) of
// the four 32-token groups of K or V page j of sequence `cur`, in two steps so
// that no arithmetic waits on a load where the loads are issued:
// page_lookup loads the page's slot (from the plan's slots -- sparse with a
// page table -- or the page table) into sp[0], or with P32 tables resolves the
// four sub-page indices (which needs kv_len L); page_buffers turns a looked-up
// slot into the sub-page indices.  A bad slot sets TRTV_DEVERR_PAGE_ID (the
// plan kernel has checked the plan's slots) when `flag` (one producer flags
// it) and reads slot 0.
__device__ __forceinline__ void page_lookup(const AttnParams& p, const SeqCursor& cur, int64_t j, bool sparse,
                                            bool is_v, int L, int (&sp)[kGroups]) {
  const int64_t e = static_cast<int64_t>(cur.s) * p.plan_cap + j;
  if (sparse && p.plan_slots != nullptr) {
    sp[0] = p.plan_slots[e];
    return;
  }
  const int blk = sparse ? p.plan_blocks[e] : static_cast<int>(j);
  const int64_t row = static_cast<int64_t>(cur.b) * p.max_pages + blk;
  if (p.sub_k != nullptr) {
#pragma unroll
    for (int g = 0; g < kGroups; ++g)
      sp[g] = p32_entry(is_v ? p.sub_v : p.sub_k, row * kGroups + g, blk * kGroups + g, L, p.num_subpages, p.err);
    return;
  }
  sp[0] = p.page_table[row];
}

__device__ __forceinline__ void page_buffers(const AttnParams& p, bool is_v, bool flag, int (&sp)[kGroups]) {
  if (p.sub_k != nullptr) return;  // P32 tables: resolved by page_lookup
  int slot = sp[0];
  if (slot < 0 || slot >= p.num_slots) {
    if (flag && p.plan_slots == nullptr) atomicOr(p.err, TRTV_DEVERR_PAGE_ID);
    slot = 0;
  }
  const int64_t buf = static_cast<int64_t>(slot) * p.slot_stride + (is_v ? 1 : 0);
#pragma unroll
  for (int g = 0; g < kGroups; ++g) sp[g] = static_cast<int>(buf * kGroups + g);
}

// Walk over the CTA's pages in order, across sequence ends: sequence `cur`,
// page j of its real units [j0, j1) inside the CTA's range.
struct PageWalk {
  SeqCursor cur;
  int64_t j, j0, j1;
  bool valid;
};

__device__ __forceinline__ void walk_enter(PageWalk& w, int n, bool sparse, int64_t u0, int64_t u1, int setup) {
  w.valid = (sparse ? w.cur.s : w.cur.b) < n && seq_in_range(w.cur, u1, setup);
  w.j0 = w.j = w.valid ? seq_j0(w.cur, u0, setup) : 0;
  w.j1 = w.valid ? seq_j1(w.cur, u1, setup) : 0;
}

__device__ __forceinline__ PageWalk walk_first(const int32_t* scan, int n, int Hk, bool sparse, int64_t u0,
                                               int64_t u1, int setup) {
  PageWalk w;
  w.cur = cursor_first(scan, n, Hk, sparse, u0);
  walk_enter(w, n, sparse, u0, u1, setup);
  return w;
}

// advance k pages
__device__ __forceinline__ void walk_skip(PageWalk& w, int64_t k, const int32_t* scan, int n, int Hk, bool sparse,
                                          int64_t u0, int64_t u1, int setup) {
  while (k > 0 && w.valid) {
    const int64_t rem = w.j1 - w.j;
    if (k < rem) {
      w.j += k;
      return;
    }
    k -= rem;
    cursor_next(w.cur, scan, n, Hk, sparse);
    walk_enter(w, n, sparse, u0, u1, setup);
  }
}

// Page-ahead resolution for the pages of the CTA, 32 at a time (one page per
// lane): `now` holds the current group of 32 pages, `next` the following one,
// whose loads are in flight while `now` is used -- across sequence ends, so a
// new sequence's first pages are never waited for.  (rs, rj) is the
// (sequence, page) position of the group after `next` (rs = n past the range).
struct PageAhead {
  int now[kGroups], next[kGroups];
  int rs, rj;
};

// Walk positioned at (rs, rj).
__device__ __forceinline__ PageWalk walk_at(int rs, int rj, const int32_t* scan, int n, int Hk, bool sparse,
                                            int64_t u0, int64_t u1, int setup) {
  PageWalk x;
  x.cur.s = rs;
  x.cur.b = rs / Hk;
  x.cur.h = rs % Hk;
  if (rs < n * (sparse ? 1 : Hk)) cursor_fill(x.cur, scan, Hk, sparse);
  walk_enter(x, n, sparse, u0, u1, setup);
  if (x.valid) x.j = rj;
  return x;
}

// Looks up this lane's page of the group at (rs, rj) (page_lookup); moves
// (rs, rj) on by 32 pages.
__device__ __forceinline__ void ahead_group(const AttnParams& p, int& rs, int& rj, int lane, bool sparse,
                                            bool is_v, const int32_t* scan, int n, int Hk, int64_t u0, int64_t u1,
                                            int (&sp)[kGroups]) {
#pragma unroll
  for (int g = 0; g < kGroups; ++g) sp[g] = 0;
  const int end = n * (sparse ? 1 : Hk);
  PageWalk x = walk_at(rs, rj, scan, n, Hk, sparse, u0, u1, p.setup);
  PageWalk y = x;
  walk_skip(y, lane, scan, n, Hk, sparse, u0, u1, p.setup);
  if (y.valid) {
    const int L = p.sub_k != nullptr ? p.kv_lens[y.cur.b] : 0;  // P32 tables: used entries
    page_lookup(p, y.cur, y.j, sparse, is_v, L, sp);
  }
  walk_skip(x, 32, scan, n, Hk, sparse, u0, u1, p.setup);
  rs = x.valid ? x.cur.s : end;
  rj = x.valid ? static_cast<int>(x.j) : 0;
}

__device__ __forceinline__ void ahead_init(PageAhead& a, const AttnParams& p, const PageWalk& w, int lane,
                                           bool sparse, bool is_v, const int32_t* scan, int n, int Hk, int64_t u0,
                                           int64_t u1) {
  a.rs = w.valid ? w.cur.s : n * (sparse ? 1 : Hk);
  a.rj = w.valid ? static_cast<int>(w.j) : 0;
  ahead_group(p, a.rs, a.rj, lane, sparse, is_v, scan, n, Hk, u0, u1, a.now);
  ahead_group(p, a.rs, a.rj, lane, sparse, is_v, scan, n, Hk, u0, u1, a.next);
}

// after the 32 pages of `now` are used
__device__ __forceinline__ void ahead_step(PageAhead& a, const AttnParams& p, int lane, bool sparse, bool is_v,
                                           const int32_t* scan, int n, int Hk, int64_t u0, int64_t u1) {
#pragma unroll
  for (int g = 0; g < kGroups; ++g) a.now[g] = a.next[g];
  ahead_group(p, a.rs, a.rj, lane, sparse, is_v, scan, n, Hk, u0, u1, a.next);
}

// The sparse plan entries (block, token mask) of the CTA's pages for the
// softmax warps, 32 pages per group one group ahead, as PageAhead does the
// buffers for the producers.  The walk position of the group after `next` is
// kept as (sequence, page) only: the softmax holds few registers to spare.
struct PlanAhead {
  int blk_now, blk_next;
  uint32_t m_now, m_next;
  int rs, rj;
};

// Entries of group position (rs, rj) for this lane; returns the position 32
// pages on (rs = n once past the CTA's range).
__device__ __forceinline__ void plan_group(const AttnParams& p, int& rs, int& rj, int lane, const int32_t* scan,
                                           int n, int Hk, int64_t u0, int64_t u1, int& blk, uint32_t& m) {
  blk = 0;
  m = 0;
  PageWalk x = walk_at(rs, rj, scan, n, Hk, true, u0, u1, p.setup);
  PageWalk y = x;
  walk_skip(y, lane, scan, n, Hk, true, u0, u1, p.setup);
  if (y.valid) {
    const int64_t e = static_cast<int64_t>(y.cur.s) * p.plan_cap + y.j;
    blk = p.plan_blocks[e];
    m = p.plan_masks[e];
  }
  walk_skip(x, 32, scan, n, Hk, true, u0, u1, p.setup);
  rs = x.valid ? x.cur.s : n;
  rj = x.valid ? static_cast<int>(x.j) : 0;
}

__device__ __forceinline__ void plan_ahead_init(PlanAhead& a, const AttnParams& p, int lane, const int32_t* scan,
                                                int n, int Hk, int64_t u0, int64_t u1) {
  const PageWalk w = walk_first(scan, n, Hk, true, u0, u1, p.setup);
  a.rs = w.valid ? w.cur.s : n;
  a.rj = w.valid ? static_cast<int>(w.j) : 0;
  plan_group(p, a.rs, a.rj, lane, scan, n, Hk, u0, u1, a.blk_now, a.m_now);
  plan_group(p, a.rs, a.rj, lane, scan, n, Hk, u0, u1, a.blk_next, a.m_next);
}

__device__ __forceinline__ void plan_ahead_step(PlanAhead& a, const AttnParams& p, int lane, const int32_t* scan,
                                                int n, int Hk, int64_t u0, int64_t u1) {
  a.blk_now = a.blk_next;
  a.m_now = a.m_next;
  plan_group(p, a.rs, a.rj, lane, scan, n, Hk, u0, u1, a.blk_next, a.m_next);
}

template <bool FP8, int D, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ AttnParams p) {
  constexpr bool F16 = FP8;                      // mma operand type for FP8 caches
  constexpr int NB = FP8 ? 1 : (D * 2) / 128;    // TMA boxes per cache token row
  constexpr int SUBK = NB * kBox;                // bytes of one K (or V) sub-page in a stage
  constexpr int SUBV = FP8 ? 2 * kBox : SUBK;    // bytes of one V sub-page as PV reads it
  constexpr int TS = 16 * MT;                    // tokens of a page per warp
  constexpr int CH = TS < 32 ? TS : 32;          // tokens per score chunk
  constexpr int NCH = TS / CH;
  constexpr int NT = CH / 8;
  constexpr int KS = Shape<D>::KS;
  constexpr int DT = Shape<D>::DT;
  constexpr int NSL = kConsumerWarps / MT;       // token slices per page
  constexpr int HALF = D / 2 < 64 ? D / 2 : 64;  // merge columns per pass
  constexpr int MSTR = HALF + 8;                 // merge row stride (floats)
  static_assert(!FP8 || D == 128, "FP8 caches need head_dim 128");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* empty = full + p.nstages;
  int* abortf = reinterpret_cast<int*>(empty + p.nstages);  // the CTA's give-up flag
  const Waits wt{p.err, abortf, p.wait_ns};
  int32_t* scan = reinterpret_cast<int32_t*>(smem + p.off_scan);
  const bool sparse = p.sparse != 0;
  const int Hk = p.num_kv_heads, T = p.qo_len, NST = p.nstages;
  const int nitems = sparse ? p.batch * Hk : p.batch;
  int32_t* warp_tot = scan + nitems + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    *abortf = 0;
    fence_mbar_init();
  }
  pdl_wait();  // inputs may come from the previous kernel of the stream
  block_exclusive_scan(nitems, scan, warp_tot, [&](int i) -> int32_t {
    return seq_units(p, i, T, sparse);
  });
  const int64_t W = item_start(scan, nitems, Hk, sparse);
  if (threadIdx.x == 0) write_split_desc(p, scan, nitems, Hk, sparse, W);
  pdl_trigger();  // the split-combine kernel may be scheduled now
  // rows of sequences with no units (invalid request, or no selected block)
  // are zero: CTA c clears items c, c + P, ...
  for (int i = blockIdx.x; i < nitems; i += gridDim.x) {
    if (scan[i + 1] != scan[i]) continue;
    const int b = sparse ? i / Hk : i;
    const int h0 = sparse ? i % Hk : 0, nh = sparse ? 1 : Hk;
    const int span = nh * p.group * D;  // contiguous query heads of these KV heads
    for (int t = 0; t < T; ++t) {
      const int64_t o0 = ((static_cast<int64_t>(b) * T + t) * p.num_q_heads +
                          static_cast<int64_t>(h0) * p.group) * D;
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

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    prefetch_tensormap(&kv_map);
    const uint64_t pol = policy_evict_first();
    const int sub_rows = Hk * kSub;  // tensor-map rows per sub-page buffer group
    int it = 0;
    bool alive = true;
    for (SeqCursor cur = cursor_first(scan, nitems, Hk, sparse, u0);
         alive && (sparse ? cur.s : cur.b) < nitems && seq_in_range(cur, u1, p.setup);
         cursor_next(cur, scan, nitems, Hk, sparse)) {
      const int64_t j0 = seq_j0(cur, u0, p.setup), j1 = seq_j1(cur, u1, p.setup);
      const int L = p.sub_k != nullptr ? p.kv_lens[cur.b] : 0;  // P32 tables: used entries
      for (int64_t j = j0; j < j1; ++j, ++it) {
        const int st = it % NST;
        const uint32_t ph = static_cast<uint32_t>(it / NST) & 1u;
        if (p.withhold >= 0 && it >= p.withhold) { alive = false; break; }  // tests of the give-up path only
        if (it >= NST && !mbar_wait(&empty[st], ph ^ 1u, wt)) { alive = false; break; }
        const int blk = sparse ? p.plan_blocks[static_cast<int64_t>(cur.s) * p.plan_cap + j]
                               : static_cast<int>(j);
        const int64_t row = static_cast<int64_t>(cur.b) * p.max_pages + blk;
        int slot = 0;
        if (p.sub_k == nullptr) {
          slot = p.page_table[row];
          if (slot < 0 || slot >= p.num_slots) {
            atomicOr(p.err, TRTV_DEVERR_PAGE_ID);
            slot = 0;
          }
        }
        uint8_t* stage = smem + p.off_stage + st * p.stage_bytes;
        mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(p.stage_bytes));
        const int64_t kbuf = static_cast<int64_t>(slot) * p.slot_stride;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          uint8_t* dst = stage + (kv ? p.off_v : p.off_k);
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            const int sp = p.sub_k != nullptr
                               ? p32_entry(kv ? p.sub_v : p.sub_k, row * kGroups + g, blk * kGroups + g,
                                           L, p.num_subpages, p.err)
                               : static_cast<int>((kbuf + kv) * kGroups + g);
            const int y = sp * sub_rows + cur.h * kSub;
#pragma unroll
            for (int hb = 0; hb < NB; ++hb)
              tma_load_2d(dst + (g * NB + hb) * kBox, &kv_map, &full[st], hb * (FP8 ? 128 : 64), y,
                          pol);
          }
        }
      }
    }
    // never leave copies in flight: wait for the last issued pages to land
    for (int k = (it > NST ? it - NST : 0); k < it; ++k)
      mbar_drain(&full[k % NST], static_cast<uint32_t>(k / NST) & 1u, wt);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  const int mt = warp % MT, sl = warp / MT;
  const int tok0 = sl * TS;
  float* mbuf = reinterpret_cast<float*>(smem + p.off_merge);
  float* ml = reinterpret_cast<float*>(smem + p.off_ml);          // [8 warps][16 rows][2]
  float* mlf = ml + kConsumerWarps * 32;                          // [128 rows][2] final
  bool dead = false;
  int it = 0;

  for (SeqCursor cur = cursor_first(scan, nitems, Hk, sparse, u0);
       (sparse ? cur.s : cur.b) < nitems && seq_in_range(cur, u1, p.setup);
       cursor_next(cur, scan, nitems, Hk, sparse)) {
    const int b = cur.b, h = cur.h;
    const int64_t j0 = seq_j0(cur, u0, p.setup), j1 = seq_j1(cur, u1, p.setup);
    const int L = p.kv_lens[b];

    uint32_t qa[KS][4];
    load_q_frags<FP8, D>(p.q, T, p.num_q_heads, p.group, p.group_pad, b, h, mt, qa);
    int bound[2], trow[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int r = mt * 16 + g + 8 * hh;
      const int t = r / p.group_pad, gl = r % p.group_pad;
      const bool ok = t < T && gl < p.group;
      trow[hh] = ok ? t : 0;
      bound[hh] = ok ? L - T + t : -1;
    }
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    float o[DT][4];
#pragma unroll
    for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    for (int64_t j = j0; j < j1; ++j, ++it) {
      const int st = it % NST;
      const uint32_t ph = static_cast<uint32_t>(it / NST) & 1u;
      // plan entry loaded before the wait: its latency overlaps the TMA
      int blk = static_cast<int>(j);
      uint32_t tokmask = 0xffffffffu;
      if (sparse) {
        blk = p.plan_blocks[static_cast<int64_t>(cur.s) * p.plan_cap + j];
        tokmask = p.plan_masks[static_cast<int64_t>(cur.s) * p.plan_cap + j];
      }
      if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(&full[st], ph, wt));
      const int pos0 = blk * kPage;
      int bnd[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) bnd[hh] = ((tokmask >> trow[hh]) & 1u) ? bound[hh] : -1;
      const uint8_t* stage = smem + p.off_stage + st * p.stage_bytes;
      const uint8_t* kst = stage + p.off_k;
      const uint8_t* vst;
      if constexpr (FP8) {
        // convert this warp's 16 rows of V to f16 (zero past kv_len), shared by the slice
        uint8_t* conv = smem + p.off_conv + (it & 1) * (kGroups * 2 * kBox);
        const int trow0 = tok0 + mt * 16;
        const int sp = trow0 / kSub, r00 = trow0 % kSub;
        const uint8_t* vsrc = stage + p.off_v + sp * kBox;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int i = lane + 32 * q4;
          const int r = r00 + (i >> 3), ch = i & 7;
          uint4 raw = *reinterpret_cast<const uint4*>(vsrc + sw128(r, ch));
          if (pos0 + sp * kSub + r >= L) raw = make_uint4(0, 0, 0, 0);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t f[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            f[2 * k] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xffffu));
            f[2 * k + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
          }
          uint8_t* dst = conv + sp * 2 * kBox + (ch >> 2) * kBox;
          const int cb = 2 * (ch & 3);
          *reinterpret_cast<uint4*>(dst + sw128(r, cb)) = make_uint4(f[0], f[1], f[2], f[3]);
          *reinterpret_cast<uint4*>(dst + sw128(r, cb + 1)) = make_uint4(f[4], f[5], f[6], f[7]);
        }
        if (MT == 1) __syncwarp(); else named_barrier(2 + sl, MT * 32);
        vst = conv;
      } else {
        vst = stage + p.off_v;
      }

#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int ct = tok0 + cc * CH;          // chunk start within the page
        const int sp = ct / kSub, r0 = ct % kSub;
        float s[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
        // ---- S = Q K^T over the chunk
        if constexpr (FP8) {
          const uint8_t* kb = kst + sp * kBox;
#pragma unroll
          for (int jt = 0; jt < NT; ++jt) {
            const int r = r0 + 8 * jt + g;
            const uint4 w0 = *reinterpret_cast<const uint4*>(kb + sw128(r, 2 * c));
            const uint4 w1 = *reinterpret_cast<const uint4*>(kb + sw128(r, 2 * c + 1));
            const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              const uint32_t b0 = e4m3x2_to_f16x2(static_cast<uint16_t>(w[ks] & 0xffffu));
              const uint32_t b1 = e4m3x2_to_f16x2(static_cast<uint16_t>(w[ks] >> 16));
              mma16816<F16>(s[jt], qa[ks], b0, b1);
            }
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
        // ---- mask (ladder bound, selected tokens, kv_len) and online softmax.
        // Chunks wholly below the lowest ladder bound need no mask (rows
        // outside the tile see S = 0 from their zero Q and are never output).
        // The reference maximum m_r of a row moves only when the row maximum
        // grows past it by more than 8 (log2 units): P = 2^(x - m_r) stays
        // below 2^8, the division by l uses the same m_r, and O is rescaled
        // only on those rare moves.
        const bool need_mask = sparse || pos0 + ct + CH - 1 > L - T;
        float mx[2] = {-INFINITY, -INFINITY};
        if (need_mask) {
#pragma unroll
          for (int jt = 0; jt < NT; ++jt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int pos = pos0 + ct + 8 * jt + 2 * c + (e & 1);
              const float x = s[jt][e] * p.scale_log2;
              s[jt][e] = (pos <= bnd[e >> 1]) ? x : -INFINITY;
              mx[e >> 1] = fmaxf(mx[e >> 1], s[jt][e]);
            }
          }
        } else {
#pragma unroll
          for (int jt = 0; jt < NT; ++jt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              s[jt][e] *= p.scale_log2;
              mx[e >> 1] = fmaxf(mx[e >> 1], s[jt][e]);
            }
          }
        }
        float alpha[2];
        bool grow[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
          mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
          const float mc = fmaxf(m_r[hh], mx[hh]);
          grow[hh] = (m_r[hh] == -INFINITY) ? (mc != -INFINITY) : (mc > m_r[hh] + 8.0f);
          alpha[hh] = 1.f;
          if (grow[hh]) {
            alpha[hh] = (m_r[hh] == -INFINITY) ? 0.f : fast_exp2(m_r[hh] - mc);
            m_r[hh] = mc;
          }
        }
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int jt = 0; jt < NT; ++jt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float mu = m_r[e >> 1];
            s[jt][e] = (mu == -INFINITY) ? 0.f : fast_exp2(s[jt][e] - mu);
            rs[e >> 1] += s[jt][e];
          }
        }
        if (__any_sync(0xffffffffu, grow[0] || grow[1])) {
          l_r[0] *= alpha[0];
          l_r[1] *= alpha[1];
#pragma unroll
          for (int i = 0; i < DT; ++i) {
            o[i][0] *= alpha[0]; o[i][1] *= alpha[0];
            o[i][2] *= alpha[1]; o[i][3] *= alpha[1];
          }
        }
        l_r[0] += rs[0];
        l_r[1] += rs[1];
        // ---- O += P V
        const uint8_t* vb = vst + sp * SUBV;
        const bool tail = pos0 + ct + CH > L;   // rows past kv_len may hold anything
        const int mat = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int kk = 0; kk < CH / 16; ++kk) {
          uint32_t a[4];
          a[0] = pack2<F16>(s[2 * kk][0], s[2 * kk][1]);
          a[1] = pack2<F16>(s[2 * kk][2], s[2 * kk][3]);
          a[2] = pack2<F16>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
          a[3] = pack2<F16>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
          uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
          if (!FP8 && tail) {
            const int pb = pos0 + ct + 16 * kk + 2 * c;
            mlo = (pb < L ? 0x0000ffffu : 0u) | (pb + 1 < L ? 0xffff0000u : 0u);
            mhi = (pb + 8 < L ? 0x0000ffffu : 0u) | (pb + 9 < L ? 0xffff0000u : 0u);
          }
          const int r = r0 + 16 * kk + 8 * (mat & 1) + rr;
#pragma unroll
          for (int dp = 0; dp < DT / 2; ++dp) {
            const int dch = 2 * dp + (mat >> 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(smem_u32(vb + (dch >> 3) * kBox + sw128(r, dch & 7)), b0, b1, b2, b3);
            mma16816<F16>(o[2 * dp], a, b0 & mlo, b1 & mhi);
            mma16816<F16>(o[2 * dp + 1], a, b2 & mlo, b3 & mhi);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }

    // ---------------------------------------------------------- sequence end
    l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], 1);
    l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], 2);
    l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], 1);
    l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], 2);
    const bool whole = seq_whole(cur, u0, u1, p.setup);
    const int64_t slot = seq_slot(cur, u0, p.setup);
    const int64_t obase = static_cast<int64_t>(b) * T;

    if constexpr (NSL == 1) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = mt * 16 + g + 8 * hh;
        const int t = r / p.group_pad, gl = r % p.group_pad;
        if (t >= T || gl >= p.group) continue;
        const float inv = l_r[hh] > 0.f ? 1.f / l_r[hh] : 0.f;
        const float sc = whole ? inv * p.v_scale : inv;
        if (whole) {
          const int64_t orow = ((obase + t) * p.num_q_heads + static_cast<int64_t>(h) * p.group + gl) * D;
#pragma unroll
          for (int i = 0; i < DT; ++i) {
            const float v0 = o[i][2 * hh] * sc, v1 = o[i][2 * hh + 1] * sc;
            if (p.out_f32)
              *reinterpret_cast<float2*>(static_cast<float*>(p.out) + orow + 8 * i + 2 * c) = make_float2(v0, v1);
            else
              *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + orow + 8 * i + 2 * c) =
                  __floats2bfloat162_rn(v0, v1);
          }
        } else {
          float* dst = p.ws_o + (slot * p.rows_pad + r) * D;
#pragma unroll
          for (int i = 0; i < DT; ++i)
            *reinterpret_cast<float2*>(dst + 8 * i + 2 * c) = make_float2(o[i][2 * hh] * sc, o[i][2 * hh + 1] * sc);
          if (c == 0)
            p.ws_lse[slot * p.rows_pad + r] = l_r[hh] > 0.f ? m_r[hh] + __log2f(l_r[hh]) : -INFINITY;
        }
      }
    } else {
      if (c == 0) {
        ml[(warp * 16 + g) * 2 + 0] = m_r[0];
        ml[(warp * 16 + g) * 2 + 1] = l_r[0];
        ml[(warp * 16 + g + 8) * 2 + 0] = m_r[1];
        ml[(warp * 16 + g + 8) * 2 + 1] = l_r[1];
      }
      named_barrier(1, kConsumerWarps * 32);
      float f[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int rl = g + 8 * hh;
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < NSL; ++q) M = fmaxf(M, ml[((q * MT + mt) * 16 + rl) * 2]);
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float Ls = 0.f;
#pragma unroll
        for (int q = 0; q < NSL; ++q)
          Ls += ml[((q * MT + mt) * 16 + rl) * 2 + 1] * fast_exp2(ml[((q * MT + mt) * 16 + rl) * 2] - Mu);
        f[hh] = Ls > 0.f ? fast_exp2(m_r[hh] - Mu) / Ls : 0.f;
        if (sl == 0 && c == 0) {
          mlf[(mt * 16 + rl) * 2 + 0] = Mu;
          mlf[(mt * 16 + rl) * 2 + 1] = Ls;
        }
      }
#pragma unroll
      for (int half = 0; half < D / HALF; ++half) {
        for (int q = 0; q < NSL; ++q) {
          if (sl == q) {
#pragma unroll
            for (int i = 0; i < HALF / 8; ++i) {
              const int di = half * (HALF / 8) + i;
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                float2* dst = reinterpret_cast<float2*>(mbuf + (mt * 16 + g + 8 * hh) * MSTR + 8 * i + 2 * c);
                float2 v = make_float2(o[di][2 * hh] * f[hh], o[di][2 * hh + 1] * f[hh]);
                if (q != 0) { const float2 u = *dst; v.x += u.x; v.y += u.y; }
                *dst = v;
              }
            }
          }
          named_barrier(1, kConsumerWarps * 32);
        }
        // cooperative write-out of this column half (4 columns per item)
        const int tid = threadIdx.x;
        const int items = MT * 16 * (HALF / 4);
        for (int idx = tid; idx < items; idx += kConsumerWarps * 32) {
          const int r = idx / (HALF / 4), c4 = idx % (HALF / 4);
          const int t = r / p.group_pad, gl = r % p.group_pad;
          if (t >= T || gl >= p.group) continue;
          float4 v = *reinterpret_cast<const float4*>(mbuf + r * MSTR + 4 * c4);
          const int d = half * HALF + 4 * c4;
          if (whole) {
            v.x *= p.v_scale; v.y *= p.v_scale; v.z *= p.v_scale; v.w *= p.v_scale;
            const int64_t orow = ((obase + t) * p.num_q_heads + static_cast<int64_t>(h) * p.group + gl) * D;
            if (p.out_f32) {
              *reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow + d) = v;
            } else {
              __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
              uint2 pk;
              pk.x = *reinterpret_cast<uint32_t*>(&lo);
              pk.y = *reinterpret_cast<uint32_t*>(&hi);
              *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + orow + d) = pk;
            }
          } else {
            *reinterpret_cast<float4*>(p.ws_o + (slot * p.rows_pad + r) * D + d) = v;
            if (half == 0 && c4 == 0) {
              const float Mu = mlf[r * 2], Ls = mlf[r * 2 + 1];
              p.ws_lse[slot * p.rows_pad + r] = Ls > 0.f ? Mu + __log2f(Ls) : -INFINITY;
            }
          }
        }
        named_barrier(1, kConsumerWarps * 32);
      }
    }
  }
}

}  // namespace trtv
