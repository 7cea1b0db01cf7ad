// abi.cu -- the extern "C" entry points declared in include/trtv.h: argument
// validation, workspace and shared-memory planning, TMA descriptor encoding
// and kernel launches.  Host code only; it never allocates device memory,
// never synchronises (except trtv_get_device_error) and never reads device
// data, so every compute entry point can be captured into a CUDA graph.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "common.cuh"
#include "launch.h"

// Per-device error word (TRTV_DEVERR_* bits), set by the kernels.
__device__ int g_trtv_device_error;

// Scratch of trtv_verify_dense_noalloc (split-KV partials, their log-sum-exp
// and the split descriptors), resident on every device that loads the library.
constexpr size_t kNoAllocScratchBytes = size_t{24} << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace trtv {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kSmemOptin = 232448;  // opt-in shared memory per block on sm_103
constexpr size_t kAlignSlack = 1024;

std::mutex g_mu;
int g_sm_count[kMaxDevices];
int* g_err_ptr[kMaxDevices];
uint8_t* g_noalloc_ptr[kMaxDevices];
std::set<std::pair<const void*, int>> g_smem_set;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
// bounded-wait settings of the next launches (trtv_test_withhold_pages)
std::atomic<uint64_t> g_wait_ns{kWaitNs};
std::atomic<int> g_withhold{-1};

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

int sm_count() {
  const int d = current_device();
  if (d < 0) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sm_count[d] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
    g_sm_count[d] = n;
  }
  return g_sm_count[d];
}

int* err_word() {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_trtv_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<int*>(p);
  }
  return g_err_ptr[d];
}

// Device address of g_noalloc_scratch on the current device.  The host-side
// name of the array is only a stand-in: the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
uint8_t* noalloc_scratch() {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_noalloc_ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[d] = static_cast<uint8_t*>(p);
  }
  return g_noalloc_ptr[d];
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Derived shape of one call.
struct Plan {
  int group, group_pad, rows, mt, rows_pad, num_ctas, n_seq;
  int64_t pool_rows;
  // workspace
  size_t ws_o, ws_lse, ws_splits, ws_blocks, ws_masks, ws_slots, ws_count, ws_sel, ws_total;
  int plan_cap;
};

trtv_status make_plan(const trtv_geom* g, int topk, Plan* pl) {
  if (g == nullptr) return TRTV_ERR_INVALID_ARG;
  if (g->batch < 1 || g->qo_len < 1 || g->num_q_heads < 1 || g->num_kv_heads < 1 ||
      g->num_q_heads % g->num_kv_heads != 0 || g->max_pages_per_req < 1 || g->num_slots < 1 ||
      g->slot_stride < 2 || g->num_ctas < 0 || g->num_ctas > kMaxCombineParts)
    return TRTV_ERR_INVALID_ARG;
  if (g->kv_dtype != TRTV_BF16 && g->kv_dtype != TRTV_FP8_E4M3) return TRTV_ERR_INVALID_ARG;
  if (!(g->sm_scale > 0.f) || !(g->k_scale > 0.f) || !std::isfinite(g->sm_scale) ||
      !std::isfinite(g->k_scale) || !std::isfinite(g->v_scale))
    return TRTV_ERR_INVALID_ARG;
  if (g->head_dim != 64 && g->head_dim != 128) return TRTV_ERR_UNSUPPORTED;
  if (g->kv_dtype == TRTV_FP8_E4M3 && g->head_dim != 128) return TRTV_ERR_UNSUPPORTED;
  if (g->qo_len > 32) return TRTV_ERR_UNSUPPORTED;
  if (topk < 0 || topk > 1024) return TRTV_ERR_INVALID_ARG;
  Plan p{};
  p.group = g->num_q_heads / g->num_kv_heads;
  p.group_pad = p.group <= 16 ? next_pow2(p.group) : (p.group + 15) / 16 * 16;
  p.rows = p.group_pad * g->qo_len;
  p.mt = next_pow2((p.rows + 15) / 16);
  if (p.mt > 8) return TRTV_ERR_UNSUPPORTED;
  p.rows_pad = 16 * p.mt;
  p.pool_rows = static_cast<int64_t>(g->num_slots) * g->slot_stride * kGroups * g->num_kv_heads * kSub;
  if (p.pool_rows >= (int64_t{1} << 31)) return TRTV_ERR_UNSUPPORTED;
  p.n_seq = g->batch * g->num_kv_heads;
  if (static_cast<int64_t>(g->batch) * g->num_kv_heads > (1 << 16)) return TRTV_ERR_UNSUPPORTED;
  int ctas = g->num_ctas > 0 ? g->num_ctas : sm_count();
  if (ctas <= 0) return TRTV_ERR_CUDA;
  p.num_ctas = ctas;
  const size_t P2 = 2 * static_cast<size_t>(ctas);
  size_t off = 0;
  p.ws_o = off;
  off = align_up(off + P2 * p.rows_pad * g->head_dim * sizeof(float), 256);
  p.ws_lse = off;
  off = align_up(off + P2 * p.rows_pad * sizeof(float), 256);
  p.ws_splits = off;
  off = align_up(off + static_cast<size_t>(ctas) * sizeof(SplitDesc), 256);
  p.plan_cap = topk > 0 ? std::min(g->qo_len * topk, g->max_pages_per_req) : 0;
  p.ws_blocks = off;
  off = align_up(off + static_cast<size_t>(p.n_seq) * p.plan_cap * sizeof(int32_t), 256);
  p.ws_masks = off;
  off = align_up(off + static_cast<size_t>(p.n_seq) * p.plan_cap * sizeof(uint32_t), 256);
  p.ws_slots = off;
  off = align_up(off + static_cast<size_t>(p.n_seq) * p.plan_cap * sizeof(int32_t), 256);
  p.ws_count = off;
  off = align_up(off + (topk > 0 ? static_cast<size_t>(p.n_seq) * sizeof(int32_t) : 0), 256);
  p.ws_sel = off;  // fused proxy + top-k: pages done per sequence
  off = align_up(off + (topk > 0 ? static_cast<size_t>(p.n_seq) * sizeof(int32_t) : 0), 256);
  p.ws_total = off;
  *pl = p;
  return TRTV_OK;
}

// The sparse plan's regions of the workspace (slots only with a page table).
PlanOut plan_out(const Plan& pl, uint8_t* wsb, bool slots) {
  PlanOut o;
  o.blocks = reinterpret_cast<int32_t*>(wsb + pl.ws_blocks);
  o.masks = reinterpret_cast<uint32_t*>(wsb + pl.ws_masks);
  o.count = reinterpret_cast<int32_t*>(wsb + pl.ws_count);
  o.slots = slots ? reinterpret_cast<int32_t*>(wsb + pl.ws_slots) : nullptr;
  o.cap = pl.plan_cap;
  return o;
}

bool encode_pool_map(const trtv_geom* g, const Plan& pl, const void* pool, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (enc == nullptr) return false;
  const bool fp8 = g->kv_dtype == TRTV_FP8_E4M3;
  const int elem = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(g->head_dim), static_cast<cuuint64_t>(pl.pool_rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(g->head_dim) * elem};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem), 32};
  cuuint32_t estr[2] = {1, 1};
  std::memset(map, 0, sizeof(*map));
  const CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                         const_cast<void*>(pool), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Shared-memory carve-up of the attention kernel; false if it cannot fit.
bool plan_attn_smem(const trtv_geom* g, const Plan& pl, bool sparse, AttnParams* a, size_t* bytes) {
  const bool fp8 = g->kv_dtype == TRTV_FP8_E4M3;
  const int D = g->head_dim;
  const int NB = fp8 ? 1 : D * 2 / 128;
  const int nsl = kConsumerWarps / pl.mt;
  const int half = D / 2 < 64 ? D / 2 : 64;
  const size_t stage = static_cast<size_t>(2) * kGroups * NB * kBox;
  const size_t conv = fp8 ? static_cast<size_t>(2) * kGroups * 2 * kBox : 0;
  const size_t merge = nsl > 1 ? static_cast<size_t>(pl.mt) * 16 * (half + 8) * sizeof(float) : 0;
  const size_t ml = (kConsumerWarps * 16 * 2 + 128 * 2) * sizeof(float);
  const int nitems = sparse ? pl.n_seq : g->batch;
  const size_t scan = align_up((static_cast<size_t>(nitems) + 1 + 32) * sizeof(int32_t), 16);
  const size_t budget = kSmemOptin - kAlignSlack;
  const size_t fixed = conv + merge + ml + scan + 2 * 8 * sizeof(uint64_t);
  if (fixed + 2 * stage > budget) return false;
  int nst = static_cast<int>((budget - fixed) / stage);
  if (nst > 4) nst = 4;
  size_t off = 0;
  a->off_stage = 0;
  a->stage_bytes = static_cast<int>(stage);
  a->off_k = 0;
  a->off_v = static_cast<int>(stage / 2);
  off = static_cast<size_t>(nst) * stage;
  a->off_conv = static_cast<int>(off);
  off += conv;
  a->off_merge = static_cast<int>(off);
  off += merge;
  a->off_ml = static_cast<int>(off);
  off += ml;
  a->off_scan = static_cast<int>(off);
  off += scan;
  a->off_bar = static_cast<int>(align_up(off, 8));
  off = a->off_bar + 2 * nst * sizeof(uint64_t) + 8;  // barriers, give-up flag
  a->nstages = nst;
  *bytes = off + kAlignSlack;
  return *bytes <= kSmemOptin;
}

// 3-D view of q [B*T][Hq][D] for the tcgen05 proxy's Q tiles: box [T][G][64].
bool encode_q_map(const trtv_geom* g, const Plan& pl, const void* q, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(g->head_dim), static_cast<cuuint64_t>(g->num_q_heads),
                        static_cast<cuuint64_t>(g->batch) * g->qo_len};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(g->head_dim) * 2,
                           static_cast<cuuint64_t>(g->num_q_heads) * g->head_dim * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(pl.group), static_cast<cuuint32_t>(g->qo_len)};
  cuuint32_t estr[3] = {1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The row-major tcgen05 attention kernel covers head_dim 128 and a
// power-of-two group: bf16 caches with 32 < group * qo_len <= 128 rows (one
// UMMA M = 128 tile; below 33 rows the mma.sync kernel keeps pace with the
// HBM stream), FP8 caches with 32 < group * qo_len <= 64 (E4M3 UMMAs read the
// pages as they are; the lane quadrants without rows host the warps that
// quantise Q; tiles of at most 32 rows go to the position-major kernel).
bool attn_umma_eligible(const trtv_geom* g, const Plan& pl, const void* q) {
  if (g->head_dim != 128 || pl.group != pl.group_pad || !aligned(q, 16)) return false;
  const int rows = pl.group * g->qo_len;
  if (g->kv_dtype == TRTV_FP8_E4M3) return rows > 32 && rows <= 64;
  return rows > 32 && rows <= 128;
}

bool plan_attn_umma_smem(const trtv_geom* g, const Plan& pl, bool sparse, AttnParams* a, size_t* bytes) {
  const bool fp8 = g->kv_dtype == TRTV_FP8_E4M3;
  // Q tile (as TMA writes it): rows x 128 head dims of bf16 in two 64-column
  // halves; at most 64 rows take 16 KB (the M = 128 UMMA then reads rows
  // 64..127 from whatever follows the tile into accumulator rows nobody reads)
  const size_t qbuf = pl.group * g->qo_len <= 64 ? 64 * 128 * 2 : 128 * 128 * 2;
  // FP8: the two E4M3 terms of Q (64 rows x 128 B each), right before the K ring
  const size_t qf8 = fp8 ? 2 * 64 * 128 : 0;
  const size_t kv = fp8 ? static_cast<size_t>(kGroups) * kBox : static_cast<size_t>(kGroups) * 2 * kBox;
  const int nitems = sparse ? pl.n_seq : g->batch;
  const size_t scan = align_up((static_cast<size_t>(nitems) + 1 + 32) * sizeof(int32_t), 16);
  const size_t ml = 1280 * sizeof(float);
  const int nq = kUmmaAttnQTiles;
  // bf16: K stages are freed by QK, V stages only by PV, so V gets its depth
  // first and a third K stage comes when it fits.  FP8: equal rings of 16 KB
  // stages, as deep as fit.
  for (int depth = fp8 ? kUmmaAttnFp8Stages : kUmmaAttnKStagesMax; depth >= 2; --depth) {
    const int nk = depth, nv = fp8 ? depth : kUmmaAttnVStages;
    size_t off = 0;
    a->off_q = 0;
    off += nq * qbuf;
    a->off_qf8 = static_cast<int>(off);
    off += qf8;
    a->off_stage = static_cast<int>(off);
    a->stage_bytes = static_cast<int>(kv);
    off += nk * kv;
    a->off_vring = static_cast<int>(off);
    off += nv * kv;
    a->off_scan = static_cast<int>(off);
    off += scan;
    a->off_ml = static_cast<int>(off);
    off += ml;
    a->off_bar = static_cast<int>(align_up(off, 8));
    off = a->off_bar + (2 * nk + 2 * nv + 24) * sizeof(uint64_t) + 16;
    a->nstages = nk;
    a->nv = nv;
    a->nq = nq;
    a->qbuf = static_cast<int>(qbuf);
    a->off_k = a->off_v = a->off_conv = a->off_merge = 0;
    *bytes = off + kAlignSlack;
    if (*bytes <= kSmemOptin) return true;
  }
  return false;
}

// The position-major tcgen05 kernel (positions on the UMMA's M, rows on N)
// covers FP8 caches with head_dim 128 and a power-of-two group with at most 32
// rows (group * qo_len): the FP8 verify and drafter tiles, where rows as M
// would leave most of each instruction idle.  (Its bf16 form keeps up with the
// HBM stream too, but racing ahead of the mma.sync kernel's pace it leaves
// some SMs with less bandwidth and a longer tail, so bf16 tiles of at most 32
// rows stay on the mma.sync kernel.)
bool attn_pm_eligible(const trtv_geom* g, const Plan& pl, const void* q) {
  return g->kv_dtype == TRTV_FP8_E4M3 && g->head_dim == 128 && pl.group == pl.group_pad && aligned(q, 16) &&
         pl.group * g->qo_len <= 32;
}

// Shared memory of the position-major kernel: Q tiles (bf16, two 64-column
// halves of rows_pad rows), FP8: two sequences' E4M3 Q terms, the P^T regions
// (four buffers of 2 rows_pad bytes per 128-byte row), the K and V rings; as
// deep as fits, two Q tiles preferred.
bool plan_attn_pm_smem(const trtv_geom* g, const Plan& pl, bool sparse, AttnParams* a, size_t* bytes) {
  const bool fp8 = g->kv_dtype == TRTV_FP8_E4M3;
  const int nr = pl.rows_pad;
  const size_t qbuf = static_cast<size_t>(2) * nr * 128;
  const size_t qf8 = fp8 ? static_cast<size_t>(2) * 2 * nr * 128 : 0;
  const size_t preg = static_cast<size_t>(128 * 128) * nr / 16;  // four P^T buffers of 2 nr bytes per row
  const size_t kv = fp8 ? static_cast<size_t>(kGroups) * kBox : static_cast<size_t>(kGroups) * 2 * kBox;
  const int nitems = sparse ? pl.n_seq : g->batch;
  const size_t scan = align_up((static_cast<size_t>(nitems) + 1 + 32) * sizeof(int32_t), 16);
  const size_t ml = static_cast<size_t>(8 + 4 + 2) * nr * sizeof(float) + 8 * sizeof(int);  // + vote slots
  struct Depth { int nq, nk, nv; };
  static const Depth kBf16[] = {{2, 3, 3}, {1, 3, 3}, {2, 3, 2}, {2, 2, 2}};
  static const Depth kFp8[] = {{2, 6, 6}, {2, 6, 5}, {2, 5, 5}, {2, 5, 4}, {2, 4, 4}, {2, 3, 3}, {2, 2, 2}};
  const Depth* list = fp8 ? kFp8 : kBf16;
  const int nlist = fp8 ? 7 : 4;
  for (int i = 0; i < nlist; ++i) {
    const Depth d = list[i];
    size_t off = 0;
    a->off_q = 0;
    off += d.nq * qbuf;
    a->off_qf8 = static_cast<int>(off);
    off += qf8;
    a->off_p = static_cast<int>(off);
    off += preg;
    a->off_stage = static_cast<int>(off);
    a->stage_bytes = static_cast<int>(kv);
    off += d.nk * kv;
    a->off_vring = static_cast<int>(off);
    off += d.nv * kv;
    a->off_scan = static_cast<int>(off);
    off += scan;
    a->off_ml = static_cast<int>(align_up(off, 16));
    off = a->off_ml + ml;
    a->off_bar = static_cast<int>(align_up(off, 8));
    off = a->off_bar + (2 * d.nk + 2 * d.nv + 24) * sizeof(uint64_t) + 16;
    a->nstages = d.nk;
    a->nv = d.nv;
    a->nq = d.nq;
    a->np = 4;
    a->qbuf = static_cast<int>(qbuf);
    a->off_k = a->off_v = a->off_conv = a->off_merge = 0;
    *bytes = off + kAlignSlack;
    if (*bytes <= kSmemOptin) return true;
  }
  return false;
}

// The tcgen05 proxy covers bf16, head_dim 128, a power-of-two group <= 16 with
// group * qo_len <= 128 rows (one UMMA M = 128 tile).
bool proxy_umma_eligible(const trtv_geom* g, const Plan& pl, const void* q) {
  return g->kv_dtype == TRTV_BF16 && g->head_dim == 128 && pl.group == pl.group_pad &&
         pl.group <= 16 && pl.group * g->qo_len <= 128 && aligned(q, 16);
}

// fused: room for the fused top-k's histograms (8 warps x 1 KB).
bool plan_proxy_umma_smem(const trtv_geom* g, const Plan& pl, bool fused, ProxyParams* a, size_t* bytes) {
  const size_t qbuf = pl.group * g->qo_len <= 64 ? 64 * 128 * 2 : 128 * 128 * 2;
  const size_t qbufs = 2 * qbuf;
  const size_t hist = fused ? 8 * 256 * sizeof(uint32_t) : 0;
  const size_t stage = static_cast<size_t>(kGroups) * 2 * kBox;
  const size_t scan = align_up((static_cast<size_t>(g->batch) + 1 + 32) * sizeof(int32_t), 16);
  const size_t budget = kSmemOptin - kAlignSlack - 1024;
  const size_t fixed = qbufs + hist + scan + (2 * 8 + 9) * sizeof(uint64_t) + 16;
  if (fixed + 2 * stage > budget) return false;
  int nst = static_cast<int>((budget - fixed) / stage);
  if (nst > 6) nst = 6;
  a->off_q = 0;
  a->qbuf = static_cast<int>(qbuf);
  a->off_stage = static_cast<int>(qbufs);
  a->stage_bytes = static_cast<int>(stage);
  size_t off = qbufs + static_cast<size_t>(nst) * stage;
  a->off_red = static_cast<int>(off);
  off += hist;
  a->off_scan = static_cast<int>(off);
  off += scan;
  a->off_bar = static_cast<int>(align_up(off, 8));
  off = a->off_bar + (2 * nst + 9) * sizeof(uint64_t) + 16;
  a->nstages = nst;
  *bytes = off + kAlignSlack;
  return *bytes <= kSmemOptin - 1024;
}

bool plan_proxy_smem(const trtv_geom* g, const Plan& pl, ProxyParams* a, size_t* bytes) {
  const bool fp8 = g->kv_dtype == TRTV_FP8_E4M3;
  const int NB = fp8 ? 1 : g->head_dim * 2 / 128;
  const size_t stage = static_cast<size_t>(kGroups) * NB * kBox;
  const size_t scan = align_up((static_cast<size_t>(g->batch) + 1 + 32) * sizeof(int32_t), 16);
  const size_t budget = kSmemOptin - kAlignSlack - 1024;  // 1 KB for static shared memory
  const size_t per_stage = stage + 8 * 32 * sizeof(float) + 2 * sizeof(uint64_t);
  if (scan + 2 * per_stage > budget) return false;
  int nst = static_cast<int>((budget - scan) / per_stage);
  if (nst > 8) nst = 8;
  (void)pl;
  size_t off = 0;
  a->off_stage = 0;
  a->stage_bytes = static_cast<int>(stage);
  off = static_cast<size_t>(nst) * stage;
  a->off_red = static_cast<int>(off);
  off += static_cast<size_t>(nst) * 8 * 32 * sizeof(float);
  a->off_scan = static_cast<int>(off);
  off += scan;
  a->off_bar = static_cast<int>(align_up(off, 8));
  off = a->off_bar + 2 * nst * sizeof(uint64_t) + 8;  // barriers, give-up flag
  a->nstages = nst;
  *bytes = off + kAlignSlack;
  return *bytes <= kSmemOptin - 1024;
}

// How the attention kernels find a request's pages: a padded P128 table, a
// flat table rebuilt into the workspace first, or the P32 sub-page tables.
struct KvIndex {
  const int32_t* page_table;
  const int32_t* flat;
  const int32_t* k_sub;
  const int32_t* v_sub;
};

size_t flat_table_bytes(const trtv_geom* g) {
  return align_up(static_cast<size_t>(g->batch) * g->max_pages_per_req * sizeof(int32_t), 256);
}

bool flat_geometry_ok(const trtv_geom* g) {
  return static_cast<int64_t>(g->batch) * g->max_pages_per_req < (int64_t{1} << 31) &&
         g->batch <= 65536;
}

// plan_ready (sparse): the workspace already holds this call's sparse plan
// (the fused select built it), so the plan kernel is skipped.
trtv_status attn_common(const trtv_geom* g, const void* q, const void* pool, const KvIndex& kvi,
                        const int32_t* lens, const int32_t* block_idx, int topk, void* out,
                        int32_t out_dtype, void* ws, size_t ws_bytes, void* stream, bool plan_ready = false) {
  const bool sparse = block_idx != nullptr;
  const bool p32 = kvi.k_sub != nullptr || kvi.v_sub != nullptr;
  Plan pl;
  trtv_status s = make_plan(g, sparse ? topk : 0, &pl);
  if (s != TRTV_OK) return s;
  if (sparse && topk < 1) return TRTV_ERR_INVALID_ARG;
  const int32_t* pt = kvi.flat != nullptr ? kvi.flat : kvi.page_table;
  if (p32 ? (kvi.k_sub == nullptr || kvi.v_sub == nullptr) : pt == nullptr) return TRTV_ERR_INVALID_ARG;
  if (q == nullptr || pool == nullptr || lens == nullptr || out == nullptr)
    return TRTV_ERR_INVALID_ARG;
  if (out_dtype != TRTV_BF16 && out_dtype != TRTV_F32) return TRTV_ERR_INVALID_ARG;
  if (!aligned(pool, 16) || !aligned(q, 8) || !aligned(out, out_dtype == TRTV_F32 ? 16 : 8))
    return TRTV_ERR_INVALID_ARG;
  if (kvi.flat != nullptr && !flat_geometry_ok(g)) return TRTV_ERR_UNSUPPORTED;
  const size_t ws_need = pl.ws_total + (kvi.flat != nullptr ? flat_table_bytes(g) : 0);
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < ws_need) return TRTV_ERR_WORKSPACE;
  if (sparse && g->max_pages_per_req > 16384) return TRTV_ERR_UNSUPPORTED;
  int* err = err_word();
  if (err == nullptr) return TRTV_ERR_CUDA;
  AttnParams a{};
  size_t smem = 0;
  const bool pm = attn_pm_eligible(g, pl, q);
  const bool umma = !pm && attn_umma_eligible(g, pl, q);
  if (pm ? !plan_attn_pm_smem(g, pl, sparse, &a, &smem)
         : umma ? !plan_attn_umma_smem(g, pl, sparse, &a, &smem) : !plan_attn_smem(g, pl, sparse, &a, &smem))
    return TRTV_ERR_UNSUPPORTED;
  CUtensorMap map, qmap;
  if (!encode_pool_map(g, pl, pool, &map)) return TRTV_ERR_CUDA;
  if ((pm || umma) && !encode_q_map(g, pl, q, &qmap)) return TRTV_ERR_CUDA;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  a.q = static_cast<const __nv_bfloat16*>(q);
  // the flat table's padded form goes to the workspace after the call's own regions
  int32_t* rebuilt = kvi.flat != nullptr ? reinterpret_cast<int32_t*>(wsb + pl.ws_total) : nullptr;
  a.page_table = p32 ? nullptr : (rebuilt != nullptr ? rebuilt : kvi.page_table);
  a.sub_k = kvi.k_sub;
  a.sub_v = kvi.v_sub;
  a.num_subpages = static_cast<int>(static_cast<int64_t>(g->num_slots) * g->slot_stride * kGroups);
  a.kv_lens = lens;
  a.out = out;
  a.ws_o = reinterpret_cast<float*>(wsb + pl.ws_o);
  a.ws_lse = reinterpret_cast<float*>(wsb + pl.ws_lse);
  a.splits = reinterpret_cast<SplitDesc*>(wsb + pl.ws_splits);
  a.plan_blocks = sparse ? reinterpret_cast<const int32_t*>(wsb + pl.ws_blocks) : nullptr;
  a.plan_masks = sparse ? reinterpret_cast<const uint32_t*>(wsb + pl.ws_masks) : nullptr;
  a.plan_count = sparse ? reinterpret_cast<const int32_t*>(wsb + pl.ws_count) : nullptr;
  a.plan_slots = sparse && !p32 ? reinterpret_cast<const int32_t*>(wsb + pl.ws_slots) : nullptr;
  a.err = err;
  a.batch = g->batch;
  a.qo_len = g->qo_len;
  a.num_q_heads = g->num_q_heads;
  a.num_kv_heads = g->num_kv_heads;
  a.group = pl.group;
  a.group_pad = pl.group_pad;
  a.head_dim = g->head_dim;
  a.max_pages = g->max_pages_per_req;
  a.num_slots = g->num_slots;
  a.slot_stride = g->slot_stride;
  a.rows = pl.rows;
  a.rows_pad = pl.rows_pad;
  a.plan_cap = pl.plan_cap;
  a.sparse = sparse ? 1 : 0;
  a.out_f32 = out_dtype == TRTV_F32 ? 1 : 0;
  a.num_ctas = pl.num_ctas;
  a.scale_log2 = g->sm_scale * g->k_scale * 1.4426950408889634f;
  a.v_scale = g->v_scale;
  // stream-K charge per sequence start, in pages: what a sequence switch costs
  // each kernel relative to one page of K and V
  a.setup = pm ? kPmSeqSetup : umma ? kUmmaSeqSetup : kSeqSetup;
  a.lg_group = 0;
  while ((1 << a.lg_group) < pl.group) ++a.lg_group;
  a.wait_ns = g_wait_ns.load();
  a.withhold = g_withhold.load();
  cudaError_t e;
  if (rebuilt != nullptr) {
    e = launch_flat_table(false, kvi.flat, lens, g->batch, g->qo_len, g->max_pages_per_req, rebuilt,
                          nullptr, err, st);
    if (e != cudaSuccess) return TRTV_ERR_CUDA;
  }
  if (sparse && !plan_ready) {
    e = launch_sparse_plan(block_idx, lens, g->batch, g->qo_len, g->num_kv_heads, g->max_pages_per_req, topk,
                           plan_out(pl, wsb, !p32), a.page_table, g->num_slots, err, st);
    if (e != cudaSuccess) return TRTV_ERR_CUDA;
  }
  e = pm     ? launch_attn_pm(g->kv_dtype == TRTV_FP8_E4M3, pl.rows_pad, map, qmap, a, pl.num_ctas, smem, st)
      : umma ? (g->kv_dtype == TRTV_FP8_E4M3 ? launch_attn_umma_fp8(map, qmap, a, pl.num_ctas, smem, st)
                                           : launch_attn_umma(map, qmap, a, pl.num_ctas, smem, st))
       : g->kv_dtype == TRTV_FP8_E4M3
           ? launch_attn_fp8(g->head_dim, pl.mt, map, a, pl.num_ctas, smem, st)
           : launch_attn_bf16(g->head_dim, pl.mt, map, a, pl.num_ctas, smem, st);
  if (e != cudaSuccess) return TRTV_ERR_CUDA;
  e = launch_combine(g->head_dim, a, st);
  return e == cudaSuccess ? TRTV_OK : TRTV_ERR_CUDA;
}

}  // namespace

cudaError_t ensure_smem_attr(const void* func, size_t bytes) {
  const int d = current_device();
  if (d < 0) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_smem_set.count({func, d})) return cudaSuccess;
  }
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, func);
  if (e != cudaSuccess) return e;
  if (bytes + fa.sharedSizeBytes > kSmemOptin) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemOptin - fa.sharedSizeBytes));
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  g_smem_set.insert({func, d});
  return cudaSuccess;
}

}  // namespace trtv

using namespace trtv;

extern "C" {

const char* trtv_status_string(trtv_status s) {
  switch (s) {
    case TRTV_OK: return "ok";
    case TRTV_ERR_INVALID_ARG: return "invalid argument";
    case TRTV_ERR_UNSUPPORTED: return "unsupported geometry";
    case TRTV_ERR_CUDA: return "CUDA error";
    case TRTV_ERR_WORKSPACE: return "workspace too small or misaligned";
  }
  return "unknown status";
}

int32_t trtv_version(void) { return 100; }

size_t trtv_workspace_bytes(const trtv_geom* geom, int32_t topk) {
  Plan pl;
  if (make_plan(geom, topk, &pl) != TRTV_OK) return 0;
  return pl.ws_total;
}

trtv_status trtv_subpage_view(const trtv_geom* g, const int32_t* page_table, const int32_t* kv_lens,
                              int32_t* k_sub, int32_t* v_sub, void* stream) {
  if (g == nullptr || page_table == nullptr || kv_lens == nullptr || k_sub == nullptr ||
      v_sub == nullptr)
    return TRTV_ERR_INVALID_ARG;
  if (g->batch < 1 || g->qo_len < 1 || g->max_pages_per_req < 1 || g->num_slots < 1 ||
      g->slot_stride < 2)
    return TRTV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(g->num_slots) * g->slot_stride * kGroups + kGroups >= (int64_t{1} << 31))
    return TRTV_ERR_UNSUPPORTED;
  int* err = err_word();
  if (err == nullptr) return TRTV_ERR_CUDA;
  const cudaError_t e = launch_subpage_view(page_table, kv_lens, k_sub, v_sub, g->batch, g->qo_len,
                                            g->max_pages_per_req, g->num_slots, g->slot_stride, err,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TRTV_OK : TRTV_ERR_CUDA;
}

trtv_status trtv_verify_dense(const trtv_geom* geom, const void* q, const void* kv_pool,
                              const int32_t* page_table, const int32_t* kv_lens, void* out,
                              int32_t out_dtype, void* workspace, size_t ws_bytes, void* stream) {
  return attn_common(geom, q, kv_pool, KvIndex{page_table, nullptr, nullptr, nullptr}, kv_lens, nullptr,
                     0, out, out_dtype, workspace, ws_bytes, stream);
}

trtv_status trtv_verify_dense_noalloc(const trtv_geom* geom, const void* q, const void* kv_pool,
                                      const int32_t* page_table, const int32_t* kv_lens, void* out,
                                      int32_t out_dtype, void* stream) {
  Plan pl;
  trtv_status s = make_plan(geom, 0, &pl);
  if (s != TRTV_OK) return s;
  if (q == nullptr || kv_pool == nullptr || page_table == nullptr || kv_lens == nullptr ||
      out == nullptr || (out_dtype != TRTV_BF16 && out_dtype != TRTV_F32))
    return TRTV_ERR_INVALID_ARG;
  if (pl.ws_total > kNoAllocScratchBytes) return TRTV_ERR_WORKSPACE;  // geometry too large
  uint8_t* ws = noalloc_scratch();
  if (ws == nullptr) return TRTV_ERR_CUDA;
  return attn_common(geom, q, kv_pool, KvIndex{page_table, nullptr, nullptr, nullptr}, kv_lens, nullptr,
                     0, out, out_dtype, ws, kNoAllocScratchBytes, stream);
}

trtv_status trtv_msa_sparse_attn(const trtv_geom* geom, const void* q, const void* kv_pool,
                                 const int32_t* page_table, const int32_t* kv_lens,
                                 const int32_t* block_idx, int32_t topk, void* out,
                                 int32_t out_dtype, void* workspace, size_t ws_bytes,
                                 void* stream) {
  if (block_idx == nullptr) return TRTV_ERR_INVALID_ARG;
  return attn_common(geom, q, kv_pool, KvIndex{page_table, nullptr, nullptr, nullptr}, kv_lens,
                     block_idx, topk, out, out_dtype, workspace, ws_bytes, stream);
}

namespace {
// Proxy scores, and with block_idx set the per-token top-k as well: fused
// into the tcgen05 proxy kernel when that kernel applies (the sequence
// counters in the workspace zeroed first), else the top-k kernel after it.
// planned (optional): when set and the fused kernel applies with at most
// kFusedPlanMaxPages pages per request, the fused kernel also builds the
// sparse plan in the workspace and *planned is set.
constexpr int kFusedPlanMaxPages = 2032;  // the plan's mask fits the histogram scratch
trtv_status proxy_common(const trtv_geom* g, const void* q, const void* kv_pool, const int32_t* page_table,
                         const int32_t* kv_lens, float* scores, int32_t topk, int32_t* block_idx, void* ws,
                         size_t ws_bytes, void* stream, bool* planned = nullptr) {
  if (planned != nullptr) *planned = false;
  const bool select = block_idx != nullptr;
  Plan pl;
  trtv_status s = make_plan(g, select ? topk : 0, &pl);
  if (s != TRTV_OK) return s;
  if (pl.group > 16) return TRTV_ERR_UNSUPPORTED;
  if (q == nullptr || kv_pool == nullptr || page_table == nullptr || kv_lens == nullptr ||
      scores == nullptr)
    return TRTV_ERR_INVALID_ARG;
  if (!aligned(kv_pool, 16) || !aligned(q, 8) || !aligned(scores, 4)) return TRTV_ERR_INVALID_ARG;
  if (select) {
    if (topk < 1 || topk > 1024) return TRTV_ERR_INVALID_ARG;
    if (g->max_pages_per_req > 16384) return TRTV_ERR_UNSUPPORTED;
    if (ws == nullptr || !aligned(ws, 256) || ws_bytes < pl.ws_total) return TRTV_ERR_WORKSPACE;
  }
  int* err = err_word();
  if (err == nullptr) return TRTV_ERR_CUDA;
  ProxyParams a{};
  size_t smem = 0;
  const bool umma = proxy_umma_eligible(g, pl, q);
  if (umma ? !plan_proxy_umma_smem(g, pl, select, &a, &smem) : !plan_proxy_smem(g, pl, &a, &smem))
    return TRTV_ERR_UNSUPPORTED;
  CUtensorMap map, qmap;
  if (!encode_pool_map(g, pl, kv_pool, &map)) return TRTV_ERR_CUDA;
  if (umma && !encode_q_map(g, pl, q, &qmap)) return TRTV_ERR_CUDA;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.page_table = page_table;
  a.kv_lens = kv_lens;
  a.scores = scores;
  a.err = err;
  a.batch = g->batch;
  a.qo_len = g->qo_len;
  a.num_q_heads = g->num_q_heads;
  a.num_kv_heads = g->num_kv_heads;
  a.group = pl.group;
  a.group_pad = pl.group_pad;
  a.head_dim = g->head_dim;
  a.max_pages = g->max_pages_per_req;
  a.num_slots = g->num_slots;
  a.slot_stride = g->slot_stride;
  a.rows = pl.rows;
  a.rows_pad = pl.rows_pad;
  a.num_ctas = pl.num_ctas;
  a.score_scale = g->sm_scale * g->k_scale;
  a.wait_ns = g_wait_ns.load();
  a.withhold = g_withhold.load();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool fused = select && umma;
  if (fused) {
    a.topk_out = block_idx;
    a.topk = topk;
    a.seq_count = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + pl.ws_sel);
    if (launch_zero(a.seq_count, pl.n_seq, st) != cudaSuccess) return TRTV_ERR_CUDA;
    if (planned != nullptr && g->max_pages_per_req <= kFusedPlanMaxPages) {
      a.plan = plan_out(pl, static_cast<uint8_t*>(ws), true);
      *planned = true;
    }
  }
  cudaError_t e = umma ? launch_proxy_umma(map, qmap, a, pl.num_ctas, smem, st)
                       : g->kv_dtype == TRTV_FP8_E4M3
                             ? launch_proxy_fp8(g->head_dim, pl.mt, map, a, pl.num_ctas, smem, st)
                             : launch_proxy_bf16(g->head_dim, pl.mt, map, a, pl.num_ctas, smem, st);
  if (e != cudaSuccess) return TRTV_ERR_CUDA;
  if (select && !fused)
    e = launch_topk(scores, kv_lens, g->batch, g->qo_len, g->num_kv_heads, g->max_pages_per_req, topk,
                    block_idx, err, st);
  return e == cudaSuccess ? TRTV_OK : TRTV_ERR_CUDA;
}
}  // namespace

trtv_status trtv_msa_proxy_score(const trtv_geom* g, const void* q, const void* kv_pool,
                                 const int32_t* page_table, const int32_t* kv_lens, float* scores,
                                 void* stream) {
  return proxy_common(g, q, kv_pool, page_table, kv_lens, scores, 0, nullptr, nullptr, 0, stream);
}

trtv_status trtv_msa_select(const trtv_geom* g, const void* q, const void* kv_pool,
                            const int32_t* page_table, const int32_t* kv_lens, int32_t topk, float* scores,
                            int32_t* block_idx, void* workspace, size_t ws_bytes, void* stream) {
  if (block_idx == nullptr) return TRTV_ERR_INVALID_ARG;
  return proxy_common(g, q, kv_pool, page_table, kv_lens, scores, topk, block_idx, workspace, ws_bytes,
                      stream);
}

trtv_status trtv_msa_verify(const trtv_geom* g, const void* q, const void* kv_pool, const int32_t* page_table,
                            const int32_t* kv_lens, int32_t topk, float* scores, int32_t* block_idx, void* out,
                            int32_t out_dtype, void* workspace, size_t ws_bytes, void* stream) {
  if (block_idx == nullptr) return TRTV_ERR_INVALID_ARG;
  bool planned = false;
  const trtv_status s = proxy_common(g, q, kv_pool, page_table, kv_lens, scores, topk, block_idx, workspace,
                                     ws_bytes, stream, &planned);
  if (s != TRTV_OK) return s;
  return attn_common(g, q, kv_pool, KvIndex{page_table, nullptr, nullptr, nullptr}, kv_lens, block_idx, topk, out,
                     out_dtype, workspace, ws_bytes, stream, planned);
}

trtv_status trtv_msa_topk(const trtv_geom* g, const float* scores, const int32_t* kv_lens,
                          int32_t topk, int32_t* block_idx, void* stream) {
  if (g == nullptr || scores == nullptr || kv_lens == nullptr || block_idx == nullptr)
    return TRTV_ERR_INVALID_ARG;
  if (g->batch < 1 || g->qo_len < 1 || g->num_kv_heads < 1 || g->max_pages_per_req < 1)
    return TRTV_ERR_INVALID_ARG;
  if (topk < 1 || topk > 1024) return TRTV_ERR_INVALID_ARG;
  if (g->max_pages_per_req > 16384) return TRTV_ERR_UNSUPPORTED;
  int* err = err_word();
  if (err == nullptr) return TRTV_ERR_CUDA;
  const cudaError_t e = launch_topk(scores, kv_lens, g->batch, g->qo_len, g->num_kv_heads,
                                    g->max_pages_per_req, topk, block_idx, err,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TRTV_OK : TRTV_ERR_CUDA;
}

trtv_status trtv_stage_kv(const trtv_geom* g, const void* k_new, const void* v_new, void* kv_pool,
                          const int32_t* page_table, const int32_t* kv_lens, void* stream) {
  Plan pl;
  trtv_status s = make_plan(g, 0, &pl);
  if (s != TRTV_OK) return s;
  if (k_new == nullptr || v_new == nullptr || kv_pool == nullptr || page_table == nullptr ||
      kv_lens == nullptr)
    return TRTV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(kv_pool, 16)) return TRTV_ERR_INVALID_ARG;
  int* err = err_word();
  if (err == nullptr) return TRTV_ERR_CUDA;
  const cudaError_t e = launch_stage_kv(k_new, v_new, kv_pool, page_table, kv_lens, g->batch, g->qo_len,
                                        g->num_kv_heads, g->head_dim, g->max_pages_per_req, g->num_slots,
                                        g->slot_stride, g->kv_dtype == TRTV_FP8_E4M3, g->k_scale,
                                        g->v_scale, err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TRTV_OK : TRTV_ERR_CUDA;
}

namespace {
trtv_status flat_table_call(bool to_flat, const trtv_geom* g, const int32_t* src, const int32_t* lens,
                            int32_t* dst, int32_t* indptr, void* stream) {
  if (g == nullptr || src == nullptr || lens == nullptr || dst == nullptr) return TRTV_ERR_INVALID_ARG;
  if (g->batch < 1 || g->qo_len < 1 || g->max_pages_per_req < 1) return TRTV_ERR_INVALID_ARG;
  if (!flat_geometry_ok(g)) return TRTV_ERR_UNSUPPORTED;
  int* err = err_word();
  if (err == nullptr) return TRTV_ERR_CUDA;
  const cudaError_t e = launch_flat_table(to_flat, src, lens, g->batch, g->qo_len, g->max_pages_per_req,
                                          dst, indptr, err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TRTV_OK : TRTV_ERR_CUDA;
}
}  // namespace

trtv_status trtv_flatten_page_table(const trtv_geom* g, const int32_t* page_table,
                                    const int32_t* kv_lens, int32_t* flat, int32_t* indptr,
                                    void* stream) {
  return flat_table_call(true, g, page_table, kv_lens, flat, indptr, stream);
}

trtv_status trtv_page_table_from_flat(const trtv_geom* g, const int32_t* flat, const int32_t* kv_lens,
                                      int32_t* page_table, void* stream) {
  return flat_table_call(false, g, flat, kv_lens, page_table, nullptr, stream);
}

size_t trtv_workspace_bytes_flat(const trtv_geom* geom) {
  Plan pl;
  if (make_plan(geom, 0, &pl) != TRTV_OK || !flat_geometry_ok(geom)) return 0;
  return pl.ws_total + flat_table_bytes(geom);
}

trtv_status trtv_verify_dense_flat(const trtv_geom* geom, const void* q, const void* kv_pool,
                                   const int32_t* flat, const int32_t* kv_lens, void* out,
                                   int32_t out_dtype, void* workspace, size_t ws_bytes,
                                   void* stream) {
  if (flat == nullptr) return TRTV_ERR_INVALID_ARG;
  return attn_common(geom, q, kv_pool, KvIndex{nullptr, flat, nullptr, nullptr}, kv_lens, nullptr, 0,
                     out, out_dtype, workspace, ws_bytes, stream);
}

trtv_status trtv_draft_attn_p32(const trtv_geom* geom, const void* q, const void* kv_pool,
                                const int32_t* k_sub, const int32_t* v_sub, const int32_t* kv_lens,
                                void* out, int32_t out_dtype, void* workspace, size_t ws_bytes,
                                void* stream) {
  if (k_sub == nullptr || v_sub == nullptr) return TRTV_ERR_INVALID_ARG;
  return attn_common(geom, q, kv_pool, KvIndex{nullptr, nullptr, k_sub, v_sub}, kv_lens, nullptr, 0,
                     out, out_dtype, workspace, ws_bytes, stream);
}

trtv_status trtv_test_withhold_pages(int32_t pages, uint32_t wait_us) {
  if (pages < 0) {
    g_withhold.store(-1);
    g_wait_ns.store(kWaitNs);
    return TRTV_OK;
  }
  if (wait_us == 0 || static_cast<uint64_t>(wait_us) * 1000 > kWaitNs) return TRTV_ERR_INVALID_ARG;
  g_wait_ns.store(static_cast<uint64_t>(wait_us) * 1000);
  g_withhold.store(pages);
  return TRTV_OK;
}

trtv_status trtv_get_device_error(int32_t* host_out, void* stream) {
  if (host_out == nullptr) return TRTV_ERR_INVALID_ARG;
  int* err = err_word();
  if (err == nullptr) return TRTV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return TRTV_ERR_CUDA;
  if (cudaMemsetAsync(err, 0, sizeof(int), st) != cudaSuccess) return TRTV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return TRTV_ERR_CUDA;
  *host_out = v;
  return TRTV_OK;
}

}  // extern "C"
