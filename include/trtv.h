/*
 * trtv.h -- C ABI of the GB300 (sm_103a) verify-attention library.
 *
 * Multi-token speculative-decoding verify attention over a paged KV cache:
 * every request carries qo_len = 1 + draft_len query tokens; token t attends
 * positions p <= kv_len - qo_len + t of its request (the causal "ladder":
 * token t sees kv_len - qo_len + t + 1 positions).  Sources, by page title
 * and section:
 *   "Eagle3 for M3 MSA path + CUDA graphs compatibility" (fork PR #3),
 *     commit "... verify": the ladder, the proxy (OnlyScore) pass, top-k
 *     clipped to per-token ladder valid-page counts, sparse GQA attention;
 *     CUDA-graphs commit: device-only planning, prepare-time buffers, stable
 *     pointers, kv_lens mutated on device between replays, no allocation
 *     while capturing.
 *   "wrap up eagle changes in m3 side branch" (TensorRT-LLM #18066):
 *     MiniMaxM3DraftKVCacheView commit (slot s's K page at s * stride, V page
 *     at s * stride + 1; kv_offset == 1; P128 pages) and
 *     copy_batch_block_offsets commit (padded entries address slot 0).
 *   "Default Minimax-m3 to unified draft-target kv manager" (#17835),
 *     "Grouped-HND draft KV transfer": a P128 page is consumed as four
 *     head-major 32-token groups, [group=4, local_head, 32, head_dim].
 *
 * ---- Data layout (all device memory, owned by the caller) ----------------
 *   q          bf16  [batch * qo_len, num_q_heads, head_dim]; row = b*qo_len + t
 *   kv_pool    page buffers, each [4][num_kv_heads][32][head_dim] elements of
 *              kv_dtype (bf16: 2 bytes, FP8 E4M3: 1 byte).  Slot s owns
 *              buffers s*slot_stride .. s*slot_stride + slot_stride - 1; this
 *              layer's K page is buffer s*slot_stride, its V page the next one.
 *              Position p of a request lives in slot page_table[b][p / 128],
 *              group (p % 128) / 32, row p % 32 of its head.  The pool holds
 *              num_slots * slot_stride buffers; its address must be 16-byte
 *              aligned.
 *   page_table int32 [batch, max_pages_per_req]; entries past a request's
 *              pages are ignored (conventionally 0).
 *   kv_lens    int32 [batch], read on the device at run time (may change
 *              between launches or CUDA-graph replays; never read on the host).
 *   out        [batch * qo_len, num_q_heads, head_dim] bf16 or f32.
 *   query head hq reads KV head hq / (num_q_heads / num_kv_heads).
 *
 * ---- Conventions ---------------------------------------------------------
 *   - Every entry point only validates arguments on the host and enqueues
 *     kernels on `stream` (a cudaStream_t; NULL = legacy default stream).  It
 *     never allocates, never synchronises and never reads device memory, so
 *     it may be captured into a CUDA graph; grids are sized from batch,
 *     heads and max_pages_per_req, never from kv_lens.
 *   - Returns TRTV_ERR_INVALID_ARG for inconsistent geometry or NULL
 *     pointers, TRTV_ERR_UNSUPPORTED for valid geometry outside what the
 *     kernels handle, TRTV_ERR_WORKSPACE when ws_bytes is too small, and
 *     TRTV_ERR_CUDA when a launch fails.  Nothing is enqueued on error.
 *   - Data errors are found on the device (kv_len < qo_len or beyond
 *     128 * max_pages_per_req; a used page id outside [0, num_slots) or a used
 *     P32 sub-page index outside the view; a top-k block index >=
 *     max_pages_per_req).  Affected output rows are
 *     zero (or, for a bad page id, finite but meaningless), no kernel traps,
 *     and a bit is set in a per-device error word read by
 *     trtv_get_device_error.
 *   - Calls that share a workspace must be ordered on one stream.
 */
#ifndef TRTV_H_
#define TRTV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TRTV_OK = 0,
  TRTV_ERR_INVALID_ARG = 1,
  TRTV_ERR_UNSUPPORTED = 2,
  TRTV_ERR_CUDA = 3,
  TRTV_ERR_WORKSPACE = 4
} trtv_status;

typedef enum { TRTV_BF16 = 0, TRTV_FP8_E4M3 = 1, TRTV_F32 = 2 } trtv_dtype;

/* Device error word bits (trtv_get_device_error). */
#define TRTV_DEVERR_KV_LEN 1    /* kv_len < qo_len or kv_len > 128 * max_pages */
#define TRTV_DEVERR_PAGE_ID 2   /* a used page-table entry outside [0, num_slots), or a used
                                   P32 table entry outside [0, 4 * num_slots * slot_stride) */
#define TRTV_DEVERR_BLOCK_IDX 4 /* a top-k block index >= max_pages_per_req */
#define TRTV_DEVERR_TIMEOUT 8   /* a pipeline wait gave up (2 s, or the limit set by
                                   trtv_test_withhold_pages): that call's results are invalid */

typedef struct {
  int32_t batch;             /* requests B >= 1 */
  int32_t qo_len;            /* T = 1 + draft_len, 1 <= T <= 32 */
  int32_t num_q_heads;       /* Hq */
  int32_t num_kv_heads;      /* Hk, Hq % Hk == 0 */
  int32_t head_dim;          /* D: 64 or 128 */
  int32_t max_pages_per_req; /* page-table row pitch (capacity / 128) */
  int32_t num_slots;         /* slots in the pool; page ids must be < num_slots */
  int32_t slot_stride;       /* page buffers per slot, >= 2 (V = K + 1: kv_offset == 1) */
  int32_t kv_dtype;          /* TRTV_BF16 or TRTV_FP8_E4M3 */
  float sm_scale;            /* softmax scale, e.g. 1 / sqrt(D) */
  float k_scale;             /* per-tensor dequantisation scale of K (1 for bf16) */
  float v_scale;             /* per-tensor dequantisation scale of V (1 for bf16) */
  int32_t num_ctas;          /* work CTAs of the attention / proxy kernels,
                                0..1024; 0 = one per SM.  Results depend on it
                                only through rounding (a split changes the
                                running maximum P is rounded against). */
} trtv_geom;

/* Human-readable name of a status code (static storage). */
const char* trtv_status_string(trtv_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t trtv_version(void);

/*
 * P32 sub-page view of the P128 pages (sources: #18066 view and padding
 * commits; #17835 "Grouped-HND draft KV transfer").
 * For every request b and logical 32-token block j < 4 * max_pages_per_req:
 *   s = page_table[b][j / 4] if j < ceil(kv_len[b] / 32), else 0 (padding
 *       addresses slot 0's memory);
 *   k_sub[b][j] = 4 * (s * slot_stride) + j % 4;
 *   v_sub[b][j] = 4 * (s * slot_stride + 1) + j % 4;
 * in units of one [num_kv_heads, 32, head_dim] sub-page of the pool.
 * k_sub, v_sub: int32 [batch, 4 * max_pages_per_req] device outputs.
 * Requests with bad lengths or page ids still get entries by the same rule
 * and raise the device error word.
 */
trtv_status trtv_subpage_view(const trtv_geom* geom, const int32_t* page_table,
                              const int32_t* kv_lens, int32_t* k_sub, int32_t* v_sub,
                              void* stream);

/*
 * Workspace bytes that trtv_verify_dense and trtv_msa_sparse_attn need for
 * this geometry (topk = the sparse path's k, 0 for dense only); 0 on invalid
 * geometry.  The workspace is caller-allocated device memory, 256-byte
 * aligned, with no initial contents required: every call writes each byte it
 * reads (split-KV partials, split descriptors, the sparse plan) before reading
 * it.  Calls that may overlap on the GPU must not share a workspace.
 */
size_t trtv_workspace_bytes(const trtv_geom* geom, int32_t topk);

/*
 * Dense ladder verify attention (source: PR #3 "... verify" commit; dense
 * layers' ladder SDPA mask, identical to decode at qo_len = 1).
 * out[b*T + t][hq][:] = sum_{p <= L_b - T + t} softmax_p(x) v_p, with
 *   x_p = sm_scale * k_scale * (q[b*T + t][hq] . k_p),  v_p scaled by v_scale,
 * k_p / v_p from KV head hq / G of request b.  Split-KV across CTAs; the
 * split sequences are merged by log-sum-exp in a second kernel launched on the
 * same stream; fp32 accumulation.  out_dtype: TRTV_BF16 or TRTV_F32.
 */
trtv_status trtv_verify_dense(const trtv_geom* geom, const void* q, const void* kv_pool,
                              const int32_t* page_table, const int32_t* kv_lens, void* out,
                              int32_t out_dtype, void* workspace, size_t ws_bytes,
                              void* stream);

/*
 * trtv_verify_dense without a caller-provided workspace.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory themselves -- for example a plugin whose host
 * framework owns every device allocation and hands it no allocator, or code
 * that must not call cudaMalloc between its setup and its steady state.
 * Same arguments, results and errors as trtv_verify_dense, minus workspace.
 * Scratch: one static 24 MiB device array per GPU that loads the library,
 * held until the process exits.  A geometry whose trtv_workspace_bytes(geom,
 * 0) exceeds 24 MiB is rejected with TRTV_ERR_WORKSPACE before anything is
 * enqueued.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) -- make that first call before any stream capture.
 * Every call enqueues the same kernels as trtv_verify_dense; it allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).  All calls on a device share the one array:
 * calls that may overlap on the GPU (different streams without ordering)
 * race on it and must not be issued.
 */
trtv_status trtv_verify_dense_noalloc(const trtv_geom* geom, const void* q, const void* kv_pool,
                                      const int32_t* page_table, const int32_t* kv_lens, void* out,
                                      int32_t out_dtype, void* stream);

/*
 * MSA proxy (OnlyScore) block scores (source: PR #3 "... verify" commit:
 * natively multi-token, inclusive causal bound with offset kv_len - qo_len).
 * scores[b][t][h][j] (fp32 [batch, qo_len, num_kv_heads, max_pages_per_req])
 * = max over the G query heads of KV head h and over positions p of 128-token
 * page j with p <= L_b - T + t of sm_scale * k_scale * (q . k_p); -inf for
 * pages past the bound or past the request's pages, and for every page of an
 * invalid request.  Requires G <= 16.
 */
trtv_status trtv_msa_proxy_score(const trtv_geom* geom, const void* q, const void* kv_pool,
                                 const int32_t* page_table, const int32_t* kv_lens,
                                 float* scores, void* stream);

/*
 * Per-token top-k block selection (source: PR #3 "... verify" commit: top-k
 * gets per-token ladder valid-page counts).  For each (b, t, h): of the
 * n_t = floor((L_b - T + t) / 128) + 1 blocks the token can see, keep the
 * min(topk, n_t) with the largest score, ties to the lower block index;
 * block_idx[b][t][h][0..topk) lists them in ascending order, padded with -1
 * (all -1 for an invalid request).  block_idx: int32 [B, T, Hk, topk].
 * 1 <= topk <= 1024; max_pages_per_req <= 16384.
 */
trtv_status trtv_msa_topk(const trtv_geom* geom, const float* scores, const int32_t* kv_lens,
                          int32_t topk, int32_t* block_idx, void* stream);

/*
 * Proxy scores and per-token top-k in one call (the same results as
 * trtv_msa_proxy_score followed by trtv_msa_topk; source: PR #3 "... verify"
 * commit, capture-safe device-only pipeline).  When the tcgen05 proxy kernel
 * applies (bf16 K, head_dim 128, power-of-two G <= 16, G * qo_len <= 128) the
 * top-k runs inside it: the CTA that completes the last page of a (request,
 * KV head) sequence selects that sequence's qo_len rows, so no top-k kernel
 * is launched; otherwise the top-k kernel follows the proxy kernel.
 *   scores     fp32 [B, T, Hk, max_pages] (written, as trtv_msa_proxy_score)
 *   block_idx  int32 [B, T, Hk, topk] (written, as trtv_msa_topk)
 *   workspace  >= trtv_workspace_bytes(geom, topk) bytes, 256-byte aligned; a
 *              per-sequence page counter in it is zeroed by a small kernel
 *              on `stream` before the proxy kernel (no initial contents
 *              needed).  1 <= topk <= 1024.
 * Errors as trtv_msa_proxy_score and trtv_msa_topk, plus TRTV_ERR_WORKSPACE.
 */
trtv_status trtv_msa_select(const trtv_geom* geom, const void* q, const void* kv_pool,
                            const int32_t* page_table, const int32_t* kv_lens, int32_t topk,
                            float* scores, int32_t* block_idx, void* workspace, size_t ws_bytes,
                            void* stream);

/*
 * Sparse GQA attention over the selected blocks (source: PR #3 "... verify"
 * commit).  As trtv_verify_dense, with token t of request b attending only
 * positions inside the blocks block_idx[b][t][h][0..topk) (entries < 0 are
 * ignored, repeated entries count once) and within its ladder bound.  Each
 * selected block is read once per (request, KV head) however many of the
 * request's tokens selected it.  A row with no visible position is zero.
 */
trtv_status trtv_msa_sparse_attn(const trtv_geom* geom, const void* q, const void* kv_pool,
                                 const int32_t* page_table, const int32_t* kv_lens,
                                 const int32_t* block_idx, int32_t topk, void* out,
                                 int32_t out_dtype, void* workspace, size_t ws_bytes,
                                 void* stream);

/*
 * The whole MSA verify step in one call (source: PR #3 "... verify" commit:
 * proxy scores, per-token top-k, sparse attention over the selected blocks):
 * the results of trtv_msa_select followed by trtv_msa_sparse_attn with the
 * same block_idx and topk.  When the fused select applies (see
 * trtv_msa_select) and max_pages_per_req <= 2032, the CTA that selects a
 * (request, KV head) sequence's blocks also builds the sequence's sparse plan
 * (its unique blocks, the tokens that chose each, their page slots) in the
 * workspace, and the attention runs from it: no plan kernel and no top-k
 * kernel are launched.
 *   scores     fp32 [B, T, Hk, max_pages] (written)
 *   block_idx  int32 [B, T, Hk, topk] (written)
 *   out        as trtv_msa_sparse_attn (written)
 *   workspace  >= trtv_workspace_bytes(geom, topk) bytes, 256-byte aligned,
 *              no initial contents needed.  1 <= topk <= 1024.
 * Errors as trtv_msa_select and trtv_msa_sparse_attn.
 */
trtv_status trtv_msa_verify(const trtv_geom* geom, const void* q, const void* kv_pool,
                            const int32_t* page_table, const int32_t* kv_lens, int32_t topk,
                            float* scores, int32_t* block_idx, void* out, int32_t out_dtype,
                            void* workspace, size_t ws_bytes, void* stream);

/*
 * KV slot staging along the ladder (source: PR #3 "... verify" commit: "KV
 * slot staging generalizes to the causal ladder").  Writes the K and V rows
 * of the qo_len verify tokens into their cache slots: token t of request b is
 * position p = kv_len[b] - qo_len + t, stored in slot page_table[b][p / 128]
 * at the same place the attention entry points read it (K page buffer at
 * slot * slot_stride, V at slot * slot_stride + 1, grouped-HND sub-page
 * (p % 128) / 32, row p % 32 of KV head h).
 *   k_new, v_new  bf16 [batch * qo_len, num_kv_heads, head_dim], row b*T + t,
 *                 16-byte aligned, caller-owned device memory (read only)
 *   kv_pool       the pool the attention entry points read (written)
 * bf16 caches store the bf16 bits; FP8 caches store E4M3(x / k_scale) for K
 * and E4M3(x / v_scale) for V, the quotient in binary32, rounded to nearest
 * even and saturated to +-448 (NaN stays NaN).  Nothing else of the pool is
 * written.  A request whose kv_len is invalid (< qo_len or > 128 *
 * max_pages_per_req) or whose staged page names no slot of the pool is not
 * written at all; the device error word gets TRTV_DEVERR_KV_LEN or
 * TRTV_DEVERR_PAGE_ID.  Host errors as for trtv_verify_dense.
 */
trtv_status trtv_stage_kv(const trtv_geom* geom, const void* k_new, const void* v_new, void* kv_pool,
                          const int32_t* page_table, const int32_t* kv_lens, void* stream);

/*
 * Flat (CSR) page table restaged from the padded one and the current lengths
 * (source: PR #3 "... verify" commit, "Overlap-correction fix": the flat
 * table's row layout follows the lengths, so a correction that moves a row
 * across a page boundary moves every later row and the flat table must be
 * rebuilt from the corrected lengths).  With n_b = ceil(kv_len[b] / 128)
 * (0 for kv_len <= 0, max_pages_per_req for a longer row):
 *   indptr[0] = 0,  indptr[b + 1] = indptr[b] + n_b,
 *   flat[indptr[b] + j] = page_table[b][j]  for j < n_b.
 *   page_table int32 [batch, max_pages_per_req] (read)
 *   kv_lens    int32 [batch] (read on the device)
 *   flat       int32 [batch * max_pages_per_req] (written up to indptr[batch];
 *              the rest is left as it was)
 *   indptr     int32 [batch + 1] (written), or NULL
 * Lengths outside [qo_len, 128 * max_pages_per_req] set TRTV_DEVERR_KV_LEN;
 * their rows still take n_b entries as above.  batch <= 65536.
 */
trtv_status trtv_flatten_page_table(const trtv_geom* geom, const int32_t* page_table,
                                    const int32_t* kv_lens, int32_t* flat, int32_t* indptr,
                                    void* stream);

/*
 * The consumer's side of the flat table: the padded table rebuilt on the
 * device, the row bases derived from the lengths (not an input), as above:
 *   page_table[b][j] = flat[indptr[b] + j] for j < n_b, else 0 (padding
 *   addresses slot 0, #18066 copy_batch_block_offsets commit).
 *   flat       int32, at least indptr[batch] entries (read)
 *   kv_lens    int32 [batch] (read on the device)
 *   page_table int32 [batch, max_pages_per_req] (written, every entry)
 * Errors as trtv_flatten_page_table.
 */
trtv_status trtv_page_table_from_flat(const trtv_geom* geom, const int32_t* flat,
                                      const int32_t* kv_lens, int32_t* page_table, void* stream);

/*
 * Dense ladder verify taking the flat table: trtv_page_table_from_flat into
 * the workspace, then trtv_verify_dense on it (one stream: the table
 * kernel, then the verify's kernels).
 * Workspace: trtv_workspace_bytes(geom, 0) plus
 * 4 * batch * max_pages_per_req bytes rounded up to 256
 * (trtv_workspace_bytes_flat).
 */
size_t trtv_workspace_bytes_flat(const trtv_geom* geom);
trtv_status trtv_verify_dense_flat(const trtv_geom* geom, const void* q, const void* kv_pool,
                                   const int32_t* flat, const int32_t* kv_lens, void* out,
                                   int32_t out_dtype, void* workspace, size_t ws_bytes,
                                   void* stream);

/*
 * Drafter attention through the P32 sub-page tables (sources: #17835: the
 * Eagle3 drafter consumes P32 pages of the shared P128 allocation through the
 * non-owning view; #18066 MiniMaxM3DraftKVCacheView commit: the view's index
 * scale is the draft layer's own slot stride, which may differ from a
 * pool-level page scale, e.g. 8 against 171).
 * As trtv_verify_dense (qo_len = 1 is the drafter's decode step; larger
 * qo_len applies the ladder), except that position p of KV head h of
 * request b is read from sub-page k_sub[b][p / 32] (V: v_sub[b][p / 32]) of
 * the view, element (h * 32 + p % 32) * head_dim + d of that sub-page, the
 * view's sub-page 0 being the pool's first [num_kv_heads, 32, head_dim]
 * block.  page_table is not an input: the tables may come from
 * trtv_subpage_view or from any other producer, in any order.
 *   k_sub, v_sub int32 [batch, 4 * max_pages_per_req] (read on the device);
 *                entries at or past ceil(kv_len / 32) are neither read nor
 *                checked.
 * The view spans 4 * num_slots * slot_stride sub-pages; a used entry outside
 * it sets TRTV_DEVERR_PAGE_ID and sub-page 0 is read instead (finite but
 * meaningless rows).  Workspace and other errors as trtv_verify_dense.
 */
trtv_status trtv_draft_attn_p32(const trtv_geom* geom, const void* q, const void* kv_pool,
                                const int32_t* k_sub, const int32_t* v_sub, const int32_t* kv_lens,
                                void* out, int32_t out_dtype, void* workspace, size_t ws_bytes,
                                void* stream);

/*
 * Test hook for the bounded waits (the CUDA-graphs commit of "Eagle3 for M3
 * MSA path + CUDA graphs compatibility" makes the path raise instead of
 * waiting on state that is not there; here every barrier wait inside a kernel
 * gives up after a limit, sets TRTV_DEVERR_TIMEOUT and lets the kernel return).
 *   pages >= 0: until the next call with pages < 0, in the attention and proxy
 *     kernels launched afterwards (any thread, any device) each CTA's K
 *     producer stops after `pages` pages, so the waits of its consumers run
 *     out, and every barrier wait gives up after wait_us microseconds
 *     (1 .. 2,000,000).  Outputs of those calls are invalid; no wait is left
 *     unbounded, copies already issued are waited for, TMEM is freed.
 *   pages < 0: back to normal operation (2 s bound, nothing withheld).
 * For tests only; not for production use.  TRTV_ERR_INVALID_ARG when wait_us
 * is out of range.
 */
trtv_status trtv_test_withhold_pages(int32_t pages, uint32_t wait_us);

/*
 * Read and clear the current device's error word (TRTV_DEVERR_* bits).
 * Synchronises `stream`; not for use while capturing a graph.
 */
trtv_status trtv_get_device_error(int32_t* host_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TRTV_H_ */
