/*
 * trtv_oracle.c -- plain fp64 CPU oracle for speculative-decoding verify
 * attention over a paged KV cache.  TEST INFRASTRUCTURE ONLY: the tests, the
 * package's smoke check and the benchmark's CPU-baseline leg call it; the
 * product path never does.  It shares no code, header or table with the CUDA
 * library.
 *
 * Every function is the plain definition written out, slow on purpose:
 * decode each stored element exactly to double, address it through the
 * layout rule, and evaluate the formula in the order the pages state it.
 *
 * Sources (titles of the pages; section names as they appear there):
 *  [PR18066]  "wrap up eagle changes in m3 side branch" (TensorRT-LLM #18066),
 *             commit on MiniMaxM3DraftKVCacheView: the layer-local stride puts
 *             slot s's K at s*stride and V at s*stride+1; kv_offset == 1;
 *             commit on copy_batch_block_offsets: padded entries address
 *             slot-0 memory.
 *  [PR17835]  "Default Minimax-m3 to unified draft-target kv manager"
 *             (TensorRT-LLM #17835), section "Grouped-HND draft KV transfer":
 *             a P128 page holds four head-major token groups, logically
 *             [group=4, local_head, 32, head_dim].
 *  [PR3]      "Eagle3 for M3 MSA path + CUDA graphs compatibility" (fork PR
 *             #3), commit "... verify": the verify ladder (token t of a
 *             qo_len-token row attends kv_len - qo_len + t + 1 positions), the
 *             proxy (OnlyScore) pass with inclusive causal bound
 *             offset = kv_len - qo_len, top-k limited to each token's ladder
 *             valid-page count, and sparse GQA attention over the selected
 *             blocks.
 *
 * Readings where the pages are silent:
 *  - query head hq uses KV head hq / G, G = Hq / Hk (contiguous GQA groups);
 *  - a proxy block is one 128-token page; its score is the maximum of the
 *    scaled logits over the group's query heads and the in-bound positions of
 *    the block; blocks starting past the bound score -inf;
 *  - top-k keeps min(k, n_t) blocks ordered by (score desc, index asc) and
 *    reports them in ascending index order, padded with -1;
 *  - FP8 is OCP E4M3 (bias 7, subnormals, no infinities, S.1111.111 = NaN)
 *    times the per-tensor scale;
 *  - a request with kv_len < qo_len, kv_len > 128 * max_pages, or a used page
 *    id outside [0, num_slots) is invalid: its output rows are zero and the
 *    function reports it in its return value;
 *  - the flat (CSR) page table's row b holds ceil(kv_len / 128) pages (0 for
 *    kv_len <= 0, max_pages past the capacity) from the sum of the earlier
 *    rows' counts: the row bases come from the lengths;
 *  - the drafter's attention reads K and V through the P32 tables alone; a
 *    used entry must lie in [0, 4 * num_slots * slot_stride), the view's
 *    index scale being the layer-local slot stride.
 *
 * Parity of these definitions with the pages' own implementation is not
 * checkable (the pages hold no code and no vectors); the definitions are
 * pinned by the checks in tests/oracle_pins.py (run by test_oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TRTVO_PAGE 128
#define TRTVO_SUBPAGE 32
#define TRTVO_GROUPS 4

enum { TRTVO_BF16 = 0, TRTVO_FP8_E4M3 = 1 };

/* Problem description, the oracle's own (not shared with the CUDA side). */
typedef struct {
    int32_t batch, qo_len, num_q_heads, num_kv_heads, head_dim;
    int32_t max_pages_per_req, num_slots, slot_stride, kv_dtype;
    double sm_scale, k_scale, v_scale;
} trtvo_problem;

/* ---- exact decoders ---------------------------------------------------- */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double trtvo_bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 variant: sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 is subnormal (2^-6 * m/8); the
 * single pattern S.1111.111 is NaN; there are no infinities. */
double trtvo_e4m3_to_double(uint8_t code) {
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* ---- layout ------------------------------------------------------------- */

/* Element offset (in elements of the pool) of element d of KV head h at
 * token position p of a request whose position p lives in slot `slot`.
 * kv = 0 selects the K page buffer (slot*stride), kv = 1 the V page buffer
 * (slot*stride + 1).  Within a page buffer the 128 tokens are four groups of
 * 32; group g holds [local_head][32][head_dim]. */
int64_t trtvo_element_offset(int64_t slot, int64_t stride, int64_t kv_heads, int64_t head_dim,
                             int64_t p, int64_t h, int64_t kv, int64_t d) {
    int64_t buffer = slot * stride + kv;
    int64_t in_page = p % TRTVO_PAGE;
    int64_t group = in_page / TRTVO_SUBPAGE;
    int64_t tok = in_page % TRTVO_SUBPAGE;
    int64_t buffer_elems = (int64_t)TRTVO_GROUPS * kv_heads * TRTVO_SUBPAGE * head_dim;
    int64_t group_elems = kv_heads * TRTVO_SUBPAGE * head_dim;
    return buffer * buffer_elems + group * group_elems + (h * TRTVO_SUBPAGE + tok) * head_dim + d;
}

static double load_kv(const trtvo_problem* P, const void* pool, int64_t off, int kv) {
    double scale = kv == 0 ? P->k_scale : P->v_scale;
    if (P->kv_dtype == TRTVO_FP8_E4M3)
        return trtvo_e4m3_to_double(((const uint8_t*)pool)[off]) * scale;
    return trtvo_bf16_to_double(((const uint16_t*)pool)[off]) * scale;
}

/* A request is usable when qo_len <= kv_len <= 128 * max_pages and every page
 * it touches names a slot of the pool. */
static int request_valid(const trtvo_problem* P, const int32_t* pt, const int32_t* lens, int b) {
    int32_t L = lens[b];
    if (L < P->qo_len || (int64_t)L > (int64_t)TRTVO_PAGE * P->max_pages_per_req) return 0;
    int32_t pages = (L + TRTVO_PAGE - 1) / TRTVO_PAGE;
    for (int j = 0; j < pages; ++j) {
        int32_t s = pt[(int64_t)b * P->max_pages_per_req + j];
        if (s < 0 || s >= P->num_slots) return 0;
    }
    return 1;
}

/* Contiguous copy of KV head h of request b: Kc[p][d], Vc[p][d] for
 * p < kv_len, each element decoded through the layout rule. */
static void gather_head(const trtvo_problem* P, const void* pool, const int32_t* pt,
                        int b, int L, int h, double* Kc, double* Vc) {
    int D = P->head_dim;
    for (int p = 0; p < L; ++p) {
        int64_t slot = pt[(int64_t)b * P->max_pages_per_req + p / TRTVO_PAGE];
        for (int d = 0; d < D; ++d) {
            Kc[(int64_t)p * D + d] = load_kv(P, pool,
                trtvo_element_offset(slot, P->slot_stride, P->num_kv_heads, D, p, h, 0, d), 0);
            Vc[(int64_t)p * D + d] = load_kv(P, pool,
                trtvo_element_offset(slot, P->slot_stride, P->num_kv_heads, D, p, h, 1, d), 1);
        }
    }
}

/* Public form of the gather for the tests: K and V of head h of request b as
 * [kv_len][head_dim] doubles.  Returns 0, or -1 for an invalid request. */
int trtvo_gather_head(const trtvo_problem* P, const void* pool, const int32_t* pt,
                      const int32_t* lens, int b, int h, double* Kc, double* Vc) {
    if (!request_valid(P, pt, lens, b)) return -1;
    gather_head(P, pool, pt, b, lens[b], h, Kc, Vc);
    return 0;
}

/* ---- a1: P32 sub-page view ---------------------------------------------- */

/* For logical 32-token block j of request b (j < 4 * max_pages):
 *   s = page_table[b][j / 4] while j < ceil(kv_len / 32), else slot 0
 *   k_sub[b][j] = 4 * (s * stride) + j % 4
 *   v_sub[b][j] = 4 * (s * stride + 1) + j % 4
 * in units of one [kv_heads, 32, head_dim] sub-page.  Returns the number of
 * requests whose length or used page ids are out of range (their entries
 * are still written by the same rule). */
int trtvo_subpage_view(const trtvo_problem* P, const int32_t* pt, const int32_t* lens,
                       int32_t* k_sub, int32_t* v_sub) {
    int bad = 0;
    int nsub = TRTVO_GROUPS * P->max_pages_per_req;
    for (int b = 0; b < P->batch; ++b) {
        int32_t L = lens[b];
        int64_t used = ((int64_t)L + TRTVO_SUBPAGE - 1) / TRTVO_SUBPAGE;
        if (!request_valid(P, pt, lens, b)) ++bad;
        for (int j = 0; j < nsub; ++j) {
            int64_t s = (j < used) ? pt[(int64_t)b * P->max_pages_per_req + j / TRTVO_GROUPS] : 0;
            int g = j % TRTVO_GROUPS;
            k_sub[(int64_t)b * nsub + j] = (int32_t)(TRTVO_GROUPS * (s * P->slot_stride) + g);
            v_sub[(int64_t)b * nsub + j] = (int32_t)(TRTVO_GROUPS * (s * P->slot_stride + 1) + g);
        }
    }
    return bad;
}

/* ---- a2: dense ladder verify attention ---------------------------------- */

/* Softmax attention of one query row q over positions p with keep[p] != 0,
 * p in [0, n): o = sum_p exp(x_p - max x) v_p / sum_p exp(x_p - max x),
 * x_p = sm_scale * q . k_p.  An empty set yields o = 0. */
static void attend_row(const trtvo_problem* P, const double* q, const double* Kc,
                       const double* Vc, int n, const unsigned char* keep, double* x,
                       double* o) {
    int D = P->head_dim;
    double mx = -INFINITY;
    for (int p = 0; p < n; ++p) {
        if (keep && !keep[p]) continue;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * Kc[(int64_t)p * D + d];
        x[p] = P->sm_scale * acc;
        if (x[p] > mx) mx = x[p];
    }
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (mx == -INFINITY) return;
    double den = 0.0;
    for (int p = 0; p < n; ++p) {
        if (keep && !keep[p]) continue;
        double w = exp(x[p] - mx);
        den += w;
        for (int d = 0; d < D; ++d) o[d] += w * Vc[(int64_t)p * D + d];
    }
    for (int d = 0; d < D; ++d) o[d] /= den;
}

static void load_q(const trtvo_problem* P, const uint16_t* q, int b, int t, int hq, double* out) {
    int D = P->head_dim;
    int64_t row = (int64_t)b * P->qo_len + t;
    const uint16_t* src = q + (row * P->num_q_heads + hq) * D;
    for (int d = 0; d < D; ++d) out[d] = trtvo_bf16_to_double(src[d]);
}

/* out[(b*T + t)][hq][d]: token t of request b, query head hq, attends the
 * positions p <= kv_len - qo_len + t of KV head hq / G ("token t attends
 * kv_len - qo_len + t + 1 positions", [PR3]).  Returns the number of invalid
 * requests (their rows are zero). */
int trtvo_verify_dense(const trtvo_problem* P, const uint16_t* q, const void* pool,
                       const int32_t* pt, const int32_t* lens, double* out) {
    int B = P->batch, T = P->qo_len, Hq = P->num_q_heads, Hk = P->num_kv_heads, D = P->head_dim;
    int G = Hq / Hk;
    int bad = 0;
    for (int b = 0; b < B; ++b) bad += !request_valid(P, pt, lens, b);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hk; ++bh) {
        int b = bh / Hk, h = bh % Hk;
        if (!request_valid(P, pt, lens, b)) {
            for (int t = 0; t < T; ++t)
                for (int g = 0; g < G; ++g)
                    memset(out + (((int64_t)b * T + t) * Hq + h * G + g) * D, 0, sizeof(double) * D);
            continue;
        }
        int L = lens[b];
        double* Kc = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* Vc = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* x = (double*)malloc(sizeof(double) * (size_t)L);
        double* qv = (double*)malloc(sizeof(double) * (size_t)D);
        gather_head(P, pool, pt, b, L, h, Kc, Vc);
        for (int t = 0; t < T; ++t) {
            int visible = L - T + t + 1;
            for (int g = 0; g < G; ++g) {
                int hq = h * G + g;
                load_q(P, q, b, t, hq, qv);
                attend_row(P, qv, Kc, Vc, visible, NULL, x,
                           out + (((int64_t)b * T + t) * Hq + hq) * D);
            }
        }
        free(Kc); free(Vc); free(x); free(qv);
    }
    return bad;
}

/* ---- a3: MSA proxy (OnlyScore) block scores ----------------------------- */

/* scores[b][t][h][j], j < max_pages: the maximum over the G query heads of KV
 * head h and over positions p of page j (128 j <= p <= 128 j + 127) with
 * p <= bound = kv_len - qo_len + t, of sm_scale * q . k_p; -inf when the page
 * starts past the bound.  Invalid requests score -inf everywhere.  Returns
 * the number of invalid requests. */
int trtvo_proxy_score(const trtvo_problem* P, const uint16_t* q, const void* pool,
                      const int32_t* pt, const int32_t* lens, double* scores) {
    int B = P->batch, T = P->qo_len, Hq = P->num_q_heads, Hk = P->num_kv_heads, D = P->head_dim;
    int G = Hq / Hk, NP = P->max_pages_per_req;
    int bad = 0;
    for (int b = 0; b < B; ++b) bad += !request_valid(P, pt, lens, b);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hk; ++bh) {
        int b = bh / Hk, h = bh % Hk;
        double* srow = scores + ((int64_t)b * T * Hk) * NP;
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < NP; ++j) srow[((int64_t)t * Hk + h) * NP + j] = -INFINITY;
        if (!request_valid(P, pt, lens, b)) continue;
        int L = lens[b];
        double* Kc = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* Vc = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* qv = (double*)malloc(sizeof(double) * (size_t)D);
        gather_head(P, pool, pt, b, L, h, Kc, Vc);
        for (int t = 0; t < T; ++t) {
            int bound = L - T + t;
            for (int g = 0; g < G; ++g) {
                load_q(P, q, b, t, h * G + g, qv);
                for (int p = 0; p <= bound; ++p) {
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d) acc += qv[d] * Kc[(int64_t)p * D + d];
                    double x = P->sm_scale * acc;
                    double* s = &srow[((int64_t)t * Hk + h) * NP + p / TRTVO_PAGE];
                    if (x > *s) *s = x;
                }
            }
        }
        free(Kc); free(Vc); free(qv);
    }
    return bad;
}

/* ---- a4: per-token top-k with ladder valid-page counts ------------------ */

typedef struct { double s; int32_t j; } scored_block;

static int by_score_desc_index_asc(const void* a, const void* b) {
    const scored_block* x = (const scored_block*)a;
    const scored_block* y = (const scored_block*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

static int by_index_asc(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* idx[b][t][h][0..k): of the n_t = floor(bound / 128) + 1 blocks a token can
 * see (bound = kv_len - qo_len + t), the min(k, n_t) with the largest score,
 * ties to the lower block index, listed in ascending index order and padded
 * with -1.  A request with kv_len < qo_len or beyond capacity selects nothing
 * (all -1).  Returns the number of such requests. */
int trtvo_topk(const trtvo_problem* P, const int32_t* lens, const double* scores, int k,
               int32_t* idx) {
    int B = P->batch, T = P->qo_len, Hk = P->num_kv_heads, NP = P->max_pages_per_req;
    int bad = 0;
    scored_block* cand = (scored_block*)malloc(sizeof(scored_block) * (size_t)(NP > 0 ? NP : 1));
    int32_t* pick = (int32_t*)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
    for (int b = 0; b < B; ++b) {
        int32_t L = lens[b];
        int ok = L >= T && (int64_t)L <= (int64_t)TRTVO_PAGE * NP;
        bad += !ok;
        for (int t = 0; t < T; ++t)
            for (int h = 0; h < Hk; ++h) {
                int32_t* out = idx + (((int64_t)b * T + t) * Hk + h) * k;
                for (int i = 0; i < k; ++i) out[i] = -1;
                if (!ok) continue;
                int bound = L - T + t;
                int n = bound / TRTVO_PAGE + 1;
                const double* s = scores + (((int64_t)b * T + t) * Hk + h) * NP;
                for (int j = 0; j < n; ++j) { cand[j].s = s[j]; cand[j].j = j; }
                qsort(cand, (size_t)n, sizeof(scored_block), by_score_desc_index_asc);
                int m = n < k ? n : k;
                for (int i = 0; i < m; ++i) pick[i] = cand[i].j;
                qsort(pick, (size_t)m, sizeof(int32_t), by_index_asc);
                for (int i = 0; i < m; ++i) out[i] = pick[i];
            }
    }
    free(cand); free(pick);
    return bad;
}

/* ---- a5: sparse GQA attention over the selected blocks ------------------ */

/* As the dense ladder attention, with positions further restricted to the
 * blocks listed in idx[b][t][h][0..k) (entries < 0 ignored; repeated entries
 * count once).  Returns the number of invalid requests plus the number of
 * (b, t, h) lists holding an index >= max_pages (those rows are zero). */
int trtvo_sparse_attn(const trtvo_problem* P, const uint16_t* q, const void* pool,
                      const int32_t* pt, const int32_t* lens, const int32_t* idx, int k,
                      double* out) {
    int B = P->batch, T = P->qo_len, Hq = P->num_q_heads, Hk = P->num_kv_heads, D = P->head_dim;
    int G = Hq / Hk, NP = P->max_pages_per_req;
    int bad = 0;
    for (int b = 0; b < B; ++b) bad += !request_valid(P, pt, lens, b);
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int bh = 0; bh < B * Hk; ++bh) {
        int b = bh / Hk, h = bh % Hk;
        if (!request_valid(P, pt, lens, b)) {
            for (int t = 0; t < T; ++t)
                for (int g = 0; g < G; ++g)
                    memset(out + (((int64_t)b * T + t) * Hq + h * G + g) * D, 0, sizeof(double) * D);
            continue;
        }
        int L = lens[b];
        double* Kc = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* Vc = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* x = (double*)malloc(sizeof(double) * (size_t)L);
        double* qv = (double*)malloc(sizeof(double) * (size_t)D);
        unsigned char* keep = (unsigned char*)malloc((size_t)L);
        unsigned char* chosen = (unsigned char*)malloc((size_t)NP);
        gather_head(P, pool, pt, b, L, h, Kc, Vc);
        for (int t = 0; t < T; ++t) {
            int visible = L - T + t + 1;
            const int32_t* sel = idx + (((int64_t)b * T + t) * Hk + h) * k;
            memset(chosen, 0, (size_t)NP);
            int invalid = 0;
            for (int i = 0; i < k; ++i) {
                if (sel[i] < 0) continue;
                if (sel[i] >= NP) { invalid = 1; continue; }
                chosen[sel[i]] = 1;
            }
            if (invalid) {
                ++bad;
                for (int g = 0; g < G; ++g)
                    memset(out + (((int64_t)b * T + t) * Hq + h * G + g) * D, 0, sizeof(double) * D);
                continue;
            }
            for (int p = 0; p < visible; ++p) keep[p] = chosen[p / TRTVO_PAGE];
            for (int g = 0; g < G; ++g) {
                int hq = h * G + g;
                load_q(P, q, b, t, hq, qv);
                attend_row(P, qv, Kc, Vc, visible, keep, x,
                           out + (((int64_t)b * T + t) * Hq + hq) * D);
            }
        }
        free(Kc); free(Vc); free(x); free(qv); free(keep); free(chosen);
    }
    return bad;
}

/* ---- KV slot staging along the ladder ----------------------------------- */

/* Encoding of a binary32 value as OCP E4M3 with round-to-nearest-even and
 * saturation to the largest finite magnitude (448): the finite code of the
 * same sign whose value is nearest to x; on a tie, the code with the even
 * (zero) last mantissa bit.  NaN maps to the NaN code S.1111.111; +-inf and
 * every |x| above 448 map to +-448.  Written as a search over the 127 finite
 * codes of each sign, each decoded by the definition above. */
uint8_t trtvo_e4m3_from_float(float x) {
    if (isnan(x)) return 0x7F;
    int neg = signbit(x) ? 1 : 0;
    double ax = fabs((double)x);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c < 0x7F; ++c) {          /* 0x00 .. 0x7E: +0 .. +448 */
        double v = trtvo_e4m3_to_double((uint8_t)c);
        double err = fabs(v - ax);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(best | (neg << 7));
}

/* KV slot staging ("... verify" commit of fork PR #3: KV slot staging
 * generalizes to the causal ladder).  Token t of request b is verify token t,
 * whose K and V go to position p = kv_len - qo_len + t of the request: slot
 * s = page_table[b][p / 128], element offset by the layout rule above, for
 * every KV head h and head dim d:
 *   K[p][h][d] <- k_new[b * qo_len + t][h][d],  V likewise from v_new.
 * bf16 caches store the bf16 bits unchanged.  FP8 caches store
 * E4M3(x / scale) with x the bf16 value, the quotient taken in binary32
 * (scale = k_scale for K, v_scale for V) and encoded as above.
 * A request is staged only when qo_len <= kv_len <= 128 * max_pages and the
 * page(s) holding positions kv_len - qo_len .. kv_len - 1 name slots of the
 * pool; otherwise nothing of it is written.  Returns the number of requests
 * not staged. */
int trtvo_stage_kv(const trtvo_problem* P, const uint16_t* k_new, const uint16_t* v_new,
                   const int32_t* pt, const int32_t* lens, void* pool) {
    const int T = P->qo_len, Hk = P->num_kv_heads, D = P->head_dim;
    int bad = 0;
    for (int b = 0; b < P->batch; ++b) {
        const int32_t L = lens[b];
        int ok = L >= T && (int64_t)L <= (int64_t)TRTVO_PAGE * P->max_pages_per_req;
        if (ok) {
            for (int t = 0; t < T; ++t) {
                int32_t s = pt[(int64_t)b * P->max_pages_per_req + (L - T + t) / TRTVO_PAGE];
                if (s < 0 || s >= P->num_slots) ok = 0;
            }
        }
        if (!ok) {
            ++bad;
            continue;
        }
        for (int t = 0; t < T; ++t) {
            const int64_t p = (int64_t)L - T + t;
            const int64_t slot = pt[(int64_t)b * P->max_pages_per_req + p / TRTVO_PAGE];
            for (int kv = 0; kv < 2; ++kv) {
                const uint16_t* src = kv == 0 ? k_new : v_new;
                const float scale = (float)(kv == 0 ? P->k_scale : P->v_scale);
                for (int h = 0; h < Hk; ++h)
                    for (int d = 0; d < D; ++d) {
                        const uint16_t bits = src[(((int64_t)b * T + t) * Hk + h) * D + d];
                        const int64_t off = trtvo_element_offset(slot, P->slot_stride, Hk, D, p, h, kv, d);
                        if (P->kv_dtype == TRTVO_FP8_E4M3) {
                            const float x = (float)trtvo_bf16_to_double(bits);
                            const float q = x / scale;
                            ((uint8_t*)pool)[off] = trtvo_e4m3_from_float(q);
                        } else {
                            ((uint16_t*)pool)[off] = bits;
                        }
                    }
            }
        }
    }
    return bad;
}

/* ---- f3: flat (CSR) page table rebuilt from the lengths ------------------ */

/* Pages request b occupies in the flat table: ceil(kv_len / 128), taken as 0
 * for a negative length and as max_pages for a length past the row's
 * capacity, so that every later row's base stays defined. */
static int64_t flat_pages_of(const trtvo_problem* P, int32_t L) {
    if (L <= 0) return 0;
    int64_t n = ((int64_t)L + TRTVO_PAGE - 1) / TRTVO_PAGE;
    return n > P->max_pages_per_req ? P->max_pages_per_req : n;
}

/* Restage the flat table from the padded one and the current lengths
 * ([PR3], "Overlap-correction fix": a length correction that moves a row
 * across a page boundary changes the row bases, so the flat table is rebuilt
 * from the corrected lengths):
 *   indptr[0] = 0,  indptr[b + 1] = indptr[b] + n_b,
 *   flat[indptr[b] + j] = page_table[b][j]  for j < n_b.
 * flat entries at or past indptr[batch] are left as they were; indptr may be
 * NULL.  Returns the number of requests whose length is outside
 * [qo_len, 128 * max_pages]. */
int trtvo_flatten_page_table(const trtvo_problem* P, const int32_t* pt, const int32_t* lens,
                             int32_t* flat, int32_t* indptr) {
    int bad = 0;
    int64_t base = 0;
    if (indptr) indptr[0] = 0;
    for (int b = 0; b < P->batch; ++b) {
        int32_t L = lens[b];
        if (L < P->qo_len || (int64_t)L > (int64_t)TRTVO_PAGE * P->max_pages_per_req) ++bad;
        int64_t n = flat_pages_of(P, L);
        for (int64_t j = 0; j < n; ++j) flat[base + j] = pt[(int64_t)b * P->max_pages_per_req + j];
        base += n;
        if (indptr) indptr[b + 1] = (int32_t)base;
    }
    return bad;
}

/* The consumer's side of the same layout: row b of the flat table starts at
 * sum_{b' < b} n_{b'}, computed from the lengths (the row bases are not an
 * input), and the padded table is
 *   page_table[b][j] = flat[base_b + j]  for j < n_b,  0 (slot 0) otherwise
 * (padded entries address slot 0, [PR18066]).  Returns the number of requests
 * whose length is outside [qo_len, 128 * max_pages]. */
int trtvo_page_table_from_flat(const trtvo_problem* P, const int32_t* flat, const int32_t* lens,
                               int32_t* pt) {
    int bad = 0;
    int64_t base = 0;
    for (int b = 0; b < P->batch; ++b) {
        int32_t L = lens[b];
        if (L < P->qo_len || (int64_t)L > (int64_t)TRTVO_PAGE * P->max_pages_per_req) ++bad;
        int64_t n = flat_pages_of(P, L);
        for (int64_t j = 0; j < P->max_pages_per_req; ++j)
            pt[(int64_t)b * P->max_pages_per_req + j] = j < n ? flat[base + j] : 0;
        base += n;
    }
    return bad;
}

/* ---- f4: drafter attention through the P32 sub-page tables --------------- */

/* Position p of KV head h of request b lives in sub-page k_sub[b][p / 32]
 * (V: v_sub[b][p / 32]), at element (h * 32 + p % 32) * head_dim + d of that
 * sub-page; a sub-page is one [kv_heads, 32, head_dim] block and index 0 is
 * the first sub-page of the view ([PR17835], "Grouped-HND draft KV
 * transfer"; the view's index scale is the layer-local slot stride,
 * [PR18066]).  The view spans 4 * num_slots * slot_stride sub-pages. */
static int draft_request_valid(const trtvo_problem* P, const int32_t* k_sub, const int32_t* v_sub,
                               const int32_t* lens, int b) {
    int32_t L = lens[b];
    int64_t nsub = (int64_t)TRTVO_GROUPS * P->max_pages_per_req;
    if (L < P->qo_len || (int64_t)L > (int64_t)TRTVO_SUBPAGE * nsub) return 0;
    int64_t limit = (int64_t)TRTVO_GROUPS * P->num_slots * P->slot_stride;
    int64_t used = ((int64_t)L + TRTVO_SUBPAGE - 1) / TRTVO_SUBPAGE;
    for (int64_t j = 0; j < used; ++j) {
        int64_t ks = k_sub[(int64_t)b * nsub + j], vs = v_sub[(int64_t)b * nsub + j];
        if (ks < 0 || ks >= limit || vs < 0 || vs >= limit) return 0;
    }
    return 1;
}

static void gather_head_p32(const trtvo_problem* P, const void* pool, const int32_t* k_sub,
                            const int32_t* v_sub, int b, int L, int h, double* Kc, double* Vc) {
    int D = P->head_dim;
    int64_t nsub = (int64_t)TRTVO_GROUPS * P->max_pages_per_req;
    int64_t sub_elems = (int64_t)P->num_kv_heads * TRTVO_SUBPAGE * D;
    for (int p = 0; p < L; ++p) {
        int64_t ks = k_sub[(int64_t)b * nsub + p / TRTVO_SUBPAGE];
        int64_t vs = v_sub[(int64_t)b * nsub + p / TRTVO_SUBPAGE];
        int64_t in_sub = ((int64_t)h * TRTVO_SUBPAGE + p % TRTVO_SUBPAGE) * D;
        for (int d = 0; d < D; ++d) {
            Kc[(int64_t)p * D + d] = load_kv(P, pool, ks * sub_elems + in_sub + d, 0);
            Vc[(int64_t)p * D + d] = load_kv(P, pool, vs * sub_elems + in_sub + d, 1);
        }
    }
}

/* out[(b*T + t)][hq][d]: the drafter's attention reads its KV through the P32
 * tables alone ([PR17835]: the drafter consumes P32 pages of the shared P128
 * allocation).  Query row (b, t, hq) attends positions p <= kv_len - qo_len + t
 * of KV head hq / G; qo_len = 1 is the drafter's plain decode step.  Returns
 * the number of invalid requests (length outside [qo_len, 32 * 4 * max_pages],
 * or a used sub-page index outside the view); their rows are zero. */
int trtvo_draft_attn(const trtvo_problem* P, const uint16_t* q, const void* pool,
                     const int32_t* k_sub, const int32_t* v_sub, const int32_t* lens,
                     double* out) {
    int B = P->batch, T = P->qo_len, Hq = P->num_q_heads, Hk = P->num_kv_heads, D = P->head_dim;
    int G = Hq / Hk;
    int bad = 0;
    for (int b = 0; b < B; ++b) bad += !draft_request_valid(P, k_sub, v_sub, lens, b);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hk; ++bh) {
        int b = bh / Hk, h = bh % Hk;
        if (!draft_request_valid(P, k_sub, v_sub, lens, b)) {
            for (int t = 0; t < T; ++t)
                for (int g = 0; g < G; ++g)
                    memset(out + (((int64_t)b * T + t) * Hq + h * G + g) * D, 0, sizeof(double) * D);
            continue;
        }
        int L = lens[b];
        double* Kc = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* Vc = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* x = (double*)malloc(sizeof(double) * (size_t)L);
        double* qv = (double*)malloc(sizeof(double) * (size_t)D);
        gather_head_p32(P, pool, k_sub, v_sub, b, L, h, Kc, Vc);
        for (int t = 0; t < T; ++t) {
            int visible = L - T + t + 1;
            for (int g = 0; g < G; ++g) {
                int hq = h * G + g;
                load_q(P, q, b, t, hq, qv);
                attend_row(P, qv, Kc, Vc, visible, NULL, x,
                           out + (((int64_t)b * T + t) * Hq + hq) * D);
            }
        }
        free(Kc); free(Vc); free(x); free(qv);
    }
    return bad;
}

/* Threads the OpenMP runtime will use (1 when built without OpenMP). */
int trtvo_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
