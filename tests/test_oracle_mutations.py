"""Plant plausible mistakes in copies of the oracle (on the CPU) and show that
at least one pin fails for each: the pins are strong enough to catch them."""
import pytest

import oracle
import oracle_pins

# (name, [(original text, replacement), ...]) -- each original must occur in
# the oracle source; only its first occurrence is replaced.
MUTATIONS = [
    ("ladder_off_by_one", [("int visible = L - T + t + 1;", "int visible = L - T + t;")]),
    ("proxy_bound_exclusive", [("for (int p = 0; p <= bound; ++p)", "for (int p = 0; p < bound; ++p)")]),
    ("gqa_strided_heads", [("int hq = h * G + g;", "int hq = g * Hk + h;")]),
    ("proxy_gqa_strided", [("load_q(P, q, b, t, h * G + g, qv);", "load_q(P, q, b, t, g * Hk + h, qv);")]),
    ("old_hnd_layout", [("return buffer * buffer_elems + group * group_elems + (h * TRTVO_SUBPAGE + tok) * head_dim + d;",
                         "return buffer * buffer_elems + (h * TRTVO_PAGE + in_page) * head_dim + d + 0 * group * group_elems * tok;")]),
    ("stride_ignored", [("int64_t buffer = slot * stride + kv;", "int64_t buffer = slot * 2 + kv;")]),
    ("v_before_k", [("int64_t buffer = slot * stride + kv;", "int64_t buffer = slot * stride + (1 - kv);")]),
    ("e4m3_bias_8", [("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)")]),
    ("e4m3_subnormal_scale", [("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)")]),
    ("topk_ties_to_higher", [("return (x->j > y->j) - (x->j < y->j);", "return (x->j < y->j) - (x->j > y->j);")]),
    ("topk_drops_last_valid", [("int n = bound / TRTVO_PAGE + 1;", "int n = bound / TRTVO_PAGE;")]),
    ("topk_unsorted_output", [("qsort(pick, (size_t)m, sizeof(int32_t), by_index_asc);", "(void)by_index_asc;")]),
    ("no_softmax_scale", [("x[p] = P->sm_scale * acc;", "x[p] = acc;")]),
    ("subpage_floor", [("int64_t used = ((int64_t)L + TRTVO_SUBPAGE - 1) / TRTVO_SUBPAGE;",
                        "int64_t used = (int64_t)L / TRTVO_SUBPAGE;")]),
    ("subpage_v_offset", [("k_sub[(int64_t)b * nsub + j] = (int32_t)(TRTVO_GROUPS * (s * P->slot_stride) + g);",
                           "k_sub[(int64_t)b * nsub + j] = (int32_t)(TRTVO_GROUPS * s * P->slot_stride + g * P->slot_stride);")]),
    ("sparse_ignores_ladder", [("for (int p = 0; p < visible; ++p) keep[p] = chosen[p / TRTVO_PAGE];",
                                "for (int p = 0; p < L; ++p) keep[p] = chosen[p / TRTVO_PAGE];"),
                               ("attend_row(P, qv, Kc, Vc, visible, keep, x,", "attend_row(P, qv, Kc, Vc, L, keep, x,")]),
    ("v_scale_on_k", [("double scale = kv == 0 ? P->k_scale : P->v_scale;", "double scale = kv == 0 ? P->v_scale : P->k_scale;")]),
    ("stage_position_off_by_one", [("const int64_t p = (int64_t)L - T + t;", "const int64_t p = (int64_t)L - T + t - (t == T - 1 ? 0 : -1) - 1;")]),
    ("stage_k_from_v", [("const uint16_t* src = kv == 0 ? k_new : v_new;", "const uint16_t* src = kv == 0 ? v_new : k_new;")]),
    ("stage_scale_multiplies", [("const float q = x / scale;", "const float q = x * scale;")]),
    ("stage_scales_swapped", [("const float scale = (float)(kv == 0 ? P->k_scale : P->v_scale);",
                               "const float scale = (float)(kv == 0 ? P->v_scale : P->k_scale);")]),
    ("e4m3_ties_to_lower", [("if (err < best_err || (err == best_err && (c & 1) == 0)) {", "if (err < best_err) {")]),
    ("e4m3_no_saturation", [("for (int c = 0; c < 0x7F; ++c) {", "if (ax > 448.0) return 0x7F; for (int c = 0; c < 0x7F; ++c) {")]),
    ("flat_floor_pages", [("int64_t n = ((int64_t)L + TRTVO_PAGE - 1) / TRTVO_PAGE;", "int64_t n = (int64_t)L / TRTVO_PAGE;")]),
    ("flat_padding_keeps_entry", [("j < n ? flat[base + j] : 0;", "j < n ? flat[base + j] : flat[base];")]),
    ("flat_rows_at_capacity", [("base += n;", "base += P->max_pages_per_req;")]),
    ("flat_unclamped", [("return n > P->max_pages_per_req ? P->max_pages_per_req : n;", "return n;")]),
    ("draft_k_from_v_table", [("int64_t ks = k_sub[(int64_t)b * nsub + p / TRTVO_SUBPAGE];",
                               "int64_t ks = v_sub[(int64_t)b * nsub + p / TRTVO_SUBPAGE];")]),
    ("draft_token_rotated", [("int64_t in_sub = ((int64_t)h * TRTVO_SUBPAGE + p % TRTVO_SUBPAGE) * D;",
                              "int64_t in_sub = ((int64_t)h * TRTVO_SUBPAGE + (p + 1) % TRTVO_SUBPAGE) * D;")]),
    ("draft_view_without_stride", [("int64_t limit = (int64_t)TRTVO_GROUPS * P->num_slots * P->slot_stride;",
                                    "int64_t limit = (int64_t)TRTVO_GROUPS * P->num_slots;")]),
]


@pytest.mark.parametrize("name,edits", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(name, edits):
    src = oracle.source()
    for old, new in edits:
        assert old in src, f"mutation {name}: text not found in oracle source"
        src = src.replace(old, new, 1)
    bad = oracle.load_variant(src, name)
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(bad)
        except Exception:  # any failure (assertion, invalid request) counts as caught
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
