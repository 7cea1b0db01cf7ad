"""Pins for the fp64 oracle: checks against facts fixed outside the oracle.

Every ``check_*`` takes an oracle instance (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with:

* the pages' statements, transcribed by hand into ``tests/golden/`` (ladder
  counts, ladder valid-page counts, sub-page view entries);
* published definitions evaluated by a library routine (torch's FP8/bf16
  conversions, torch's scaled-dot-product attention on contiguous K/V);
* an independent formulation of the same layout (numpy reshape/transpose of
  [group=4, local_head, 32, head_dim] page buffers instead of the oracle's
  offset arithmetic);
* closed forms and invariants (constant V, uniform logits, GQA head groups,
  same-query monotone block scores, k >= valid blocks reduces sparse to dense);
* brute force on tiny inputs (numpy block maxima, lexsorted top-k).

The same checks run against deliberately broken copies of the oracle in
``test_oracle_mutations.py`` to show that each plausible mistake fails one.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle as O
from speculative_decode_verify_kv_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------------------
# independent layout formulation (numpy reshape / transpose)

def scatter_contiguous(pool5: np.ndarray, pt: np.ndarray, stride: int, b: int,
                       K: np.ndarray, kv: int) -> None:
    """Write contiguous K[b] (shape [L, Hk, D]) into page buffers: page j of
    request b is buffer pt[b, j] * stride + kv, stored [group=4, head, 32, D]."""
    L, Hk, D = K.shape
    for j in range((L + 127) // 128):
        chunk = np.zeros((128, Hk, D), K.dtype)
        n = min(128, L - 128 * j)
        chunk[:n] = K[128 * j:128 * j + n]
        buf = chunk.reshape(4, 32, Hk, D).transpose(0, 2, 1, 3)
        sel = np.zeros((4, 32), bool)
        sel.reshape(-1)[:n] = True
        dst = pool5[pt[b, j] * stride + kv]
        for g in range(4):
            for o in range(32):
                if sel[g, o]:
                    dst[g, :, o, :] = buf[g, :, o, :]


def gather_contiguous(pool5: np.ndarray, pt: np.ndarray, stride: int, b: int, L: int,
                      kv: int) -> np.ndarray:
    """Inverse of scatter_contiguous: [L, Hk, D] raw elements."""
    _, _, Hk, _, D = pool5.shape
    out = np.zeros((L, Hk, D), pool5.dtype)
    for j in range((L + 127) // 128):
        buf = pool5[pt[b, j] * stride + kv]            # [4, Hk, 32, D]
        tok = buf.transpose(0, 2, 1, 3).reshape(128, Hk, D)
        n = min(128, L - 128 * j)
        out[128 * j:128 * j + n] = tok[:n]
    return out


def decoded(p, raw: np.ndarray, kv: int) -> np.ndarray:
    """Raw pool elements -> float64 values via torch's dtype conversion."""
    t = torch.from_numpy(np.ascontiguousarray(raw))
    if p.kv_dtype == W.FP8:
        v = t.view(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        return v * (p.k_scale if kv == 0 else p.v_scale)
    return t.view(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()


def pool5_of(p) -> np.ndarray:
    a = p.pool.contiguous()
    a = a.view(torch.int16).numpy().view(np.uint16) if a.dtype == torch.bfloat16 else a.numpy()
    return a.reshape(p.num_slots * p.slot_stride, 4, p.num_kv_heads, 32, p.head_dim)


def q64(p) -> np.ndarray:
    return p.q.to(torch.float64).numpy()          # [B*T, Hq, D]


def sdpa(qrow: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """torch scaled_dot_product_attention, float64, one query row, no mask."""
    qt = torch.from_numpy(qrow).view(1, 1, 1, -1)
    kt = torch.from_numpy(np.ascontiguousarray(K)).view(1, 1, K.shape[0], -1)
    vt = torch.from_numpy(np.ascontiguousarray(V)).view(1, 1, V.shape[0], -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale).view(-1).numpy()


def small(seed=5, lens=(5, 130, 300), T=4, Hq=8, Hk=2, D=32, stride=3, **kw):
    return W.make_problem(kv_lens=list(lens), qo_len=T, num_q_heads=Hq, num_kv_heads=Hk,
                          head_dim=D, slot_stride=stride, seed=seed, slack_slots=2, **kw)


# ---------------------------------------------------------------------------
# decoders

def check_e4m3_golden(orc):
    for code, val in _rows("e4m3.txt"):
        got = orc.e4m3_to_double(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), (code, got)


def check_e4m3_all_codes_vs_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = orc.e4m3_to_double(c)
        assert (math.isnan(got) and math.isnan(ref[c])) or got == ref[c], (hex(c), got, ref[c])


def check_bf16_all_codes_vs_torch(orc):
    codes = np.arange(0, 65536, 1, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    for c in list(range(0, 65536, 97)) + [0x3f80, 0x7f80, 0xff80, 0x0001, 0x8000, 0x7f7f]:
        got = orc.bf16_to_double(c)
        assert (math.isnan(got) and math.isnan(ref[c])) or got == ref[c], (hex(c), got)


# ---------------------------------------------------------------------------
# a1: layout and sub-page view

def check_gather_equals_independent_layout(orc):
    for stride, dtype in ((2, W.BF16), (3, W.BF16), (8, W.FP8)):
        p = small(seed=11 + stride, stride=stride, kv_dtype=dtype)
        pool5 = pool5_of(p)
        x = O.Inputs(p)
        pt = p.page_table.numpy()
        for b in range(p.batch):
            L = int(p.kv_lens[b])
            for h in range(p.num_kv_heads):
                Kc, Vc = orc.gather_head(x, b, h)
                Kr = decoded(p, gather_contiguous(pool5, pt, stride, b, L, 0)[:, h], 0)
                Vr = decoded(p, gather_contiguous(pool5, pt, stride, b, L, 1)[:, h], 1)
                assert np.array_equal(Kc, Kr) and np.array_equal(Vc, Vr), (stride, b, h)


def check_scatter_roundtrip(orc):
    """Contiguous K/V written with the independent formulation come back
    exactly through the oracle's gather (the view gathers the same bytes)."""
    p = small(seed=21, stride=2)
    rng = np.random.default_rng(3)
    pool5 = np.zeros_like(pool5_of(p))
    pt = p.page_table.numpy()
    want = {}
    for b in range(p.batch):
        L = int(p.kv_lens[b])
        for kv in (0, 1):
            vals = rng.integers(0, 0x3f00, size=(L, p.num_kv_heads, p.head_dim)).astype(np.uint16)
            scatter_contiguous(pool5, pt, 2, b, vals, kv)
            want[b, kv] = decoded(p, vals, kv)
    x = O.Inputs(p, pool=pool5)
    for b in range(p.batch):
        for h in range(p.num_kv_heads):
            Kc, Vc = orc.gather_head(x, b, h)
            assert np.array_equal(Kc, want[b, 0][:, h]) and np.array_equal(Vc, want[b, 1][:, h])


def check_old_contiguous_hnd_reading_differs(orc):
    """Reading a page as [local_head, 128, head_dim] agrees with the grouped
    layout only for head 0 in the first 32-token group ("Grouped-HND draft KV
    transfer": it selects the right heads only in the first P32 group)."""
    p = small(seed=31, lens=(256,), stride=2, Hk=2)
    pool5 = pool5_of(p)
    pt = p.page_table.numpy()
    x = O.Inputs(p)
    Kc, _ = orc.gather_head(x, 0, 0)
    Kc1, _ = orc.gather_head(x, 0, 1)
    for j in range(2):
        flat = pool5[pt[0, j] * 2].reshape(p.num_kv_heads, 128, p.head_dim)
        wrong0 = decoded(p, flat[0], 0)
        wrong1 = decoded(p, flat[1], 0)
        assert np.array_equal(Kc[128 * j:128 * j + 32], wrong0[:32])
        assert not np.array_equal(Kc[128 * j + 32:128 * j + 128], wrong0[32:])
        assert not np.array_equal(Kc1[128 * j:128 * j + 128], wrong1)


def check_subpage_view_golden(orc):
    rows = _rows("subpage_view.txt")
    i = 0
    while i < len(rows):
        assert rows[i][0] == "case"
        kw = dict(a.split("=") for a in rows[i][1:])
        stride, maxp, L = int(kw["stride"]), int(kw["max_pages"]), int(kw["kv_len"])
        row = [int(v) for v in kw["page_row"].split(",")]
        want_k = [int(v) for v in rows[i + 1][1:]]
        want_v = [int(v) for v in rows[i + 2][1:]]
        P = O.Problem(batch=1, qo_len=1, num_q_heads=1, num_kv_heads=1, head_dim=8,
                      max_pages_per_req=maxp, num_slots=max(row) + 1, slot_stride=stride,
                      kv_dtype=0, sm_scale=1.0, k_scale=1.0, v_scale=1.0)

        class X:
            pass
        x = X()
        x.P = P
        x.pt = np.array([row], np.int32)
        x.lens = np.array([L], np.int32)
        k, v, bad = orc.subpage_view(x)
        assert bad == 0
        assert k[0].tolist() == want_k and v[0].tolist() == want_v, (kw, k, v)
        i += 3


def check_subpage_view_addresses_same_elements(orc):
    """Sub-page index * sub-page size + (h*32 + p%32)*D + d is the element the
    gather reads, for every used position."""
    for stride in (2, 5):
        p = small(seed=41, stride=stride, Hk=2, D=16)
        x = O.Inputs(p)
        k, v, bad = orc.subpage_view(x)
        assert bad == 0
        sub = p.num_kv_heads * 32 * p.head_dim
        pool_flat = x.pool.reshape(-1)
        for b in range(p.batch):
            L = int(p.kv_lens[b])
            for h in range(p.num_kv_heads):
                Kc, Vc = orc.gather_head(x, b, h)
                for pos in range(L):
                    j = pos // 32
                    base = (h * 32 + pos % 32) * p.head_dim
                    ek = pool_flat[k[b, j] * sub + base: k[b, j] * sub + base + p.head_dim]
                    ev = pool_flat[v[b, j] * sub + base: v[b, j] * sub + base + p.head_dim]
                    assert np.array_equal(decoded(p, ek, 0), Kc[pos]), (stride, b, h, pos)
                    assert np.array_equal(decoded(p, ev, 1), Vc[pos]), (stride, b, h, pos)


# ---------------------------------------------------------------------------
# a2: dense ladder verify attention

def check_ladder_counts_golden(orc):
    """Uniform logits (K = 0) and V = position index: each row's output is the
    mean of its visible positions, (n - 1) / 2, which recovers n exactly."""
    for kvlen, T, t, vis in (tuple(int(v) for v in r) for r in _rows("ladder_counts.txt")):
        p = small(seed=51, lens=(kvlen,), T=T, Hq=2, Hk=1, D=8, stride=2)
        pool5 = np.zeros_like(pool5_of(p))
        pt = p.page_table.numpy()
        Vv = np.zeros((kvlen, 1, 8), np.float32)
        Vv[:, 0, 0] = np.arange(kvlen)
        Vb = torch.from_numpy(Vv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(torch.from_numpy(Vv).to(torch.bfloat16).float().numpy(), Vv)
        scatter_contiguous(pool5, pt, 2, 0, Vb, 1)
        out, bad = orc.verify_dense(O.Inputs(p, pool=pool5))
        assert bad == 0
        n = 2 * out[t, 0, 0] + 1
        assert abs(n - vis) < 1e-9, (kvlen, T, t, n, vis)


def check_dense_decode_vs_sdpa(orc):
    """qo_len = 1 is ordinary decode over all kv_len positions."""
    for dt in (W.BF16, W.FP8):
        p = small(seed=61, T=1, kv_dtype=dt, stride=2)
        out, bad = orc.verify_dense(O.Inputs(p))
        assert bad == 0
        pool5, pt, q = pool5_of(p), p.page_table.numpy(), q64(p)
        G = p.group
        for b in range(p.batch):
            L = int(p.kv_lens[b])
            K = decoded(p, gather_contiguous(pool5, pt, 2, b, L, 0), 0)
            V = decoded(p, gather_contiguous(pool5, pt, 2, b, L, 1), 1)
            for hq in range(p.num_q_heads):
                ref = sdpa(q[b, hq], K[:, hq // G], V[:, hq // G], p.sm_scale)
                assert np.allclose(out[b, hq], ref, rtol=0, atol=1e-12), (dt, b, hq)


def check_dense_ladder_rows_vs_sdpa(orc):
    """Each ladder row equals full attention over its own prefix."""
    p = small(seed=71, T=4, stride=3)
    out, bad = orc.verify_dense(O.Inputs(p))
    assert bad == 0
    pool5, pt, q = pool5_of(p), p.page_table.numpy(), q64(p)
    G, T = p.group, p.qo_len
    for b in range(p.batch):
        L = int(p.kv_lens[b])
        K = decoded(p, gather_contiguous(pool5, pt, 3, b, L, 0), 0)
        V = decoded(p, gather_contiguous(pool5, pt, 3, b, L, 1), 1)
        for t in range(T):
            n = L - T + t + 1
            for hq in range(p.num_q_heads):
                ref = sdpa(q[b * T + t, hq], K[:n, hq // G], V[:n, hq // G], p.sm_scale)
                assert np.allclose(out[b * T + t, hq], ref, rtol=0, atol=1e-12), (b, t, hq)


def check_dense_constant_v_and_gqa_groups(orc):
    """V of KV head h constant (h + 1) / 4: every query head hq outputs
    (hq // G + 1) / 4 in every component, whatever the logits."""
    p = small(seed=81, Hq=8, Hk=4, stride=2)
    pool5 = pool5_of(p).copy()
    pt = p.page_table.numpy()
    for b in range(p.batch):
        L = int(p.kv_lens[b])
        Vv = np.zeros((L, 4, p.head_dim), np.float32)
        for h in range(4):
            Vv[:, h, :] = (h + 1) / 4
        Vb = torch.from_numpy(Vv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        scatter_contiguous(pool5, pt, 2, b, Vb, 1)
    out, bad = orc.verify_dense(O.Inputs(p, pool=pool5))
    assert bad == 0
    for hq in range(8):
        assert np.allclose(out[:, hq, :], (hq // 2 + 1) / 4, rtol=0, atol=1e-12), hq


def check_dense_scales(orc):
    """FP8 per-tensor scales: k_scale multiplies the logits, v_scale the output."""
    p = small(seed=91, kv_dtype=W.FP8, stride=2)
    base, _ = orc.verify_dense(O.Inputs(p, k_scale=1.0, v_scale=1.0, sm_scale=0.25))
    scaled, _ = orc.verify_dense(O.Inputs(p, k_scale=0.5, v_scale=3.0, sm_scale=0.5))
    assert np.allclose(scaled, 3.0 * base, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# a3: proxy block scores

def _proxy_brute(p):
    pool5, pt, q = pool5_of(p), p.page_table.numpy(), q64(p)
    B, T, Hk, G, NP = p.batch, p.qo_len, p.num_kv_heads, p.group, p.max_pages_per_req
    S = np.full((B, T, Hk, NP), -np.inf)
    for b in range(B):
        L = int(p.kv_lens[b])
        K = decoded(p, gather_contiguous(pool5, pt, p.slot_stride, b, L, 0), 0)
        for t in range(T):
            bound = L - T + t
            for h in range(Hk):
                Qg = q[b * T + t, h * G:(h + 1) * G]             # [G, D]
                X = p.sm_scale * (Qg @ K[:bound + 1, h].T)       # [G, bound+1]
                for j in range(NP):
                    if 128 * j <= bound:
                        S[b, t, h, j] = X[:, 128 * j:min(128 * j + 128, bound + 1)].max()
    return S


def check_proxy_bruteforce(orc):
    for dt in (W.BF16, W.FP8):
        p = small(seed=101, lens=(4, 128, 129, 300), T=4, stride=3, kv_dtype=dt, Hq=8, Hk=2)
        S, bad = orc.proxy_score(O.Inputs(p))
        assert bad == 0
        R = _proxy_brute(p)
        assert np.array_equal(np.isinf(S), np.isinf(R))
        f = np.isfinite(R)
        assert np.allclose(S[f], R[f], rtol=0, atol=1e-12)


def check_proxy_valid_pages_golden(orc):
    for kvlen, T, t, n in (tuple(int(v) for v in r) for r in _rows("valid_pages.txt")):
        p = small(seed=111, lens=(kvlen,), T=T, Hq=4, Hk=2, D=8, stride=2)
        S, _ = orc.proxy_score(O.Inputs(p))
        finite = int(np.isfinite(S[0, t, 0]).sum())
        assert finite == n, (kvlen, T, t, finite, n)


def check_proxy_same_query_monotone(orc):
    """With the same query for every verify token, a later token sees a
    superset of positions, so its block scores are >= the earlier token's."""
    p = small(seed=121, lens=(300, 257), T=4, stride=2)
    q = p.q.view(p.batch, p.qo_len, p.num_q_heads, p.head_dim).clone()
    q[:] = q[:, :1]
    S, _ = orc.proxy_score(O.Inputs(p, q=q.view(-1, p.num_q_heads, p.head_dim)))
    for t in range(p.qo_len - 1):
        a, b = S[:, t], S[:, t + 1]
        assert np.all((b >= a) | np.isinf(a)), t
    # the last token's maximum over blocks is the largest logit of the row
    assert np.all(np.isfinite(S[:, -1, :, 0]))


# ---------------------------------------------------------------------------
# a4: top-k

def _topk_brute(lens, T, S, k):
    B, _, Hk, NP = S.shape
    idx = np.full((B, T, Hk, k), -1, np.int32)
    for b in range(B):
        L = int(lens[b])
        for t in range(T):
            n = (L - T + t) // 128 + 1
            for h in range(Hk):
                s = S[b, t, h, :n]
                order = np.lexsort((np.arange(n), -s))       # score desc, index asc
                pick = np.sort(order[:min(k, n)])
                idx[b, t, h, :len(pick)] = pick
    return idx


def check_topk_bruteforce(orc):
    rng = np.random.default_rng(7)
    p = small(seed=131, lens=(700, 1000, 129, 4), T=4, stride=2)
    p = p.with_(max_pages_per_req=8)
    pt = torch.zeros(p.batch, 8, dtype=torch.int32)
    x = O.Inputs(p, page_table=pt)
    S = rng.integers(0, 6, size=(p.batch, p.qo_len, p.num_kv_heads, 8)).astype(np.float64)
    for k in (1, 3, 5, 8, 12):
        idx, bad = orc.topk(x, S, k)
        assert bad == 0
        assert np.array_equal(idx, _topk_brute(p.kv_lens.numpy(), p.qo_len, S, k)), k


def check_topk_ties_and_clip(orc):
    p = small(seed=141, lens=(600,), T=4, stride=2).with_(max_pages_per_req=8)
    x = O.Inputs(p, page_table=torch.zeros(1, 8, dtype=torch.int32))
    S = np.zeros((1, 4, p.num_kv_heads, 8))
    S[..., 6:] = 1e30                   # past every token's bound (valid: 5 blocks)
    idx, _ = orc.topk(x, S, 3)
    assert idx[0, :, :, :].tolist() == [[[0, 1, 2]] * p.num_kv_heads] * 4
    idx, _ = orc.topk(x, S, 8)         # k >= valid blocks: all valid ones
    assert idx[0, 0, 0].tolist() == [0, 1, 2, 3, 4, -1, -1, -1]


# ---------------------------------------------------------------------------
# a5: sparse attention

def check_sparse_full_k_equals_dense(orc):
    """With k >= every token's valid-block count the selection is all valid
    blocks, and sparse attention equals dense ladder attention."""
    p = small(seed=151, lens=(300, 129, 40), T=4, stride=2)
    x = O.Inputs(p)
    S, _ = orc.proxy_score(x)
    idx, _ = orc.topk(x, S, p.max_pages_per_req)
    sp, bad = orc.sparse_attn(x, idx)
    de, _ = orc.verify_dense(x)
    assert bad == 0
    assert np.allclose(sp, de, rtol=0, atol=1e-12)


def check_sparse_single_block_vs_sdpa(orc):
    p = small(seed=161, lens=(300,), T=4, stride=2)
    x = O.Inputs(p)
    pool5, pt, q = pool5_of(p), p.page_table.numpy(), q64(p)
    L, T, G = 300, 4, p.group
    K = decoded(p, gather_contiguous(pool5, pt, 2, 0, L, 0), 0)
    V = decoded(p, gather_contiguous(pool5, pt, 2, 0, L, 1), 1)
    for blk in (0, 1, 2):
        idx = np.full((1, T, p.num_kv_heads, 3), -1, np.int32)
        idx[..., 1] = blk
        idx[..., 2] = blk                   # repeated entries count once
        out, bad = orc.sparse_attn(x, idx)
        for t in range(T):
            hi = min(128 * blk + 128, L - T + t + 1)
            for hq in range(p.num_q_heads):
                o = out[t, hq]
                if hi <= 128 * blk:
                    assert np.all(o == 0)
                    continue
                ref = sdpa(q[t, hq], K[128 * blk:hi, hq // G], V[128 * blk:hi, hq // G], p.sm_scale)
                assert np.allclose(o, ref, rtol=0, atol=1e-12), (blk, t, hq)


# ---------------------------------------------------------------------------
# KV slot staging along the ladder

def _e4m3_values():
    """Value of every finite E4M3 code via torch's float8 conversion."""
    v = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return {c: v[c] for c in range(256) if not math.isnan(v[c])}


def check_e4m3_encode_roundtrip_ties_saturation(orc):
    vals = _e4m3_values()
    for c, v in vals.items():                       # every finite code (both zeros) round-trips
        assert orc.e4m3_from_float(v) == c, (hex(c), v)
    pos = sorted((v, c) for c, v in vals.items() if c < 0x80)
    for (v0, c0), (v1, c1) in zip(pos, pos[1:]):
        mid = (v0 + v1) / 2                         # exact in binary32
        even = c0 if (c0 & 1) == 0 else c1          # ties go to the even mantissa
        assert orc.e4m3_from_float(mid) == even, (v0, v1)
        assert orc.e4m3_from_float(-mid) == even | 0x80, (v0, v1)
        below = float(np.nextafter(np.float32(mid), np.float32(-1)))
        above = float(np.nextafter(np.float32(mid), np.float32(1e9)))
        assert orc.e4m3_from_float(below) == c0 and orc.e4m3_from_float(above) == c1, (v0, v1)
    for x in (449.0, 464.0, 480.0, 1e6, float("inf")):   # saturation to +-448
        assert orc.e4m3_from_float(x) == 0x7E and orc.e4m3_from_float(-x) == 0xFE, x
    assert orc.e4m3_from_float(float("nan")) == 0x7F
    rng = np.random.default_rng(9)                  # in-range values vs torch's conversion
    xs = np.concatenate([rng.standard_normal(2000) * s for s in (1e-3, 0.1, 1.0, 30.0, 140.0)])
    xs = xs[np.abs(xs) <= 448].astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(xs, ref):
        assert orc.e4m3_from_float(float(x)) == r, (x, r)


def _staging_problem(seed, dtype, stride, lens, T=4, Hk=2, D=32, scale=None):
    kw = {}
    if scale is not None:
        kw = dict(k_scale=scale, v_scale=2 * scale)
    p = small(seed=seed, lens=lens, T=T, Hq=2 * Hk, Hk=Hk, D=D, stride=stride, kv_dtype=dtype)
    if kw:
        p = p.with_(**kw)
    g = torch.Generator().manual_seed(seed + 1)
    k_new = torch.randn(p.batch * T, Hk, D, generator=g).to(torch.bfloat16)
    v_new = torch.randn(p.batch * T, Hk, D, generator=g).to(torch.bfloat16)
    return p, k_new, v_new


def _expected_staged(p, k_new, v_new):
    """The pool after staging, written with the independent layout formulation:
    the request's tokens as contiguous [L, Hk, D] rows, the last qo_len rows
    replaced (encoded with torch's float8 conversion for FP8 caches), scattered
    back through numpy reshape / transpose."""
    pool5 = pool5_of(p).copy()
    pt = p.page_table.numpy()
    T = p.qo_len
    for b in range(p.batch):
        L = int(p.kv_lens[b])
        if L < T:
            continue
        for kv, new in ((0, k_new), (1, v_new)):
            rows = gather_contiguous(pool5, pt, p.slot_stride, b, L, kv)
            x = new[b * T:(b + 1) * T].to(torch.float32)
            if p.kv_dtype == W.FP8:
                sc = torch.tensor(p.k_scale if kv == 0 else p.v_scale, dtype=torch.float32)
                enc = (x / sc).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            else:
                enc = new[b * T:(b + 1) * T].view(torch.int16).numpy().view(np.uint16)
            rows[L - T:L] = enc
            scatter_contiguous(pool5, pt, p.slot_stride, b, rows, kv)
    return pool5


def check_stage_kv_vs_independent_layout(orc):
    for seed, dtype, stride, scale in ((31, W.BF16, 2, None), (32, W.BF16, 5, None),
                                       (33, W.FP8, 2, 0.02), (34, W.FP8, 3, 0.3)):
        p, k_new, v_new = _staging_problem(seed, dtype, stride, (5, 127, 128, 129, 300, 260), scale=scale)
        pool, bad = orc.stage_kv(O.Inputs(p), k_new, v_new)
        assert bad == 0
        want = _expected_staged(p, k_new, v_new)
        assert np.array_equal(pool.reshape(want.shape), want), (seed, dtype, stride)


def check_stage_kv_then_gather_reads_new_rows(orc):
    p, k_new, v_new = _staging_problem(35, W.BF16, 2, (7, 130))
    x = O.Inputs(p)
    pool, _ = orc.stage_kv(x, k_new, v_new)
    x2 = O.Inputs(p, pool=torch.from_numpy(pool.view(np.int16)).view(torch.bfloat16))
    T, Hk = p.qo_len, p.num_kv_heads
    for b in range(p.batch):
        L = int(p.kv_lens[b])
        for h in range(Hk):
            K0, V0 = orc.gather_head(x, b, h)
            K1, V1 = orc.gather_head(x2, b, h)
            assert np.array_equal(K1[:L - T], K0[:L - T]) and np.array_equal(V1[:L - T], V0[:L - T])
            kn = k_new[b * T:(b + 1) * T, h].to(torch.float64).numpy()
            vn = v_new[b * T:(b + 1) * T, h].to(torch.float64).numpy()
            assert np.array_equal(K1[L - T:], kn) and np.array_equal(V1[L - T:], vn), (b, h)


def check_stage_kv_fp8_saturates(orc):
    p, k_new, v_new = _staging_problem(36, W.FP8, 2, (9,), scale=0.01)
    big = torch.full_like(k_new, 100.0)             # 100 / 0.01 = 1e4 > 448
    pool, bad = orc.stage_kv(O.Inputs(p), big, -big)
    pool5 = pool.reshape(pool5_of(p).shape)
    pt = p.page_table.numpy()
    assert bad == 0
    assert np.all(gather_contiguous(pool5, pt, 2, 0, 9, 0)[5:] == 0x7E)
    assert np.all(gather_contiguous(pool5, pt, 2, 0, 9, 1)[5:] == 0xFE)


def check_stage_kv_skips_invalid_requests(orc):
    p, k_new, v_new = _staging_problem(37, W.BF16, 2, (3, 200, 40))   # kv_len 3 < qo_len 4
    pt = p.page_table.clone()
    pt[2, 0] = p.num_slots + 5                                          # staged page names no slot
    x = O.Inputs(p, page_table=pt)
    pool, bad = orc.stage_kv(x, k_new, v_new)
    assert bad == 2
    want = pool5_of(p).copy()
    exp = _expected_staged(p, k_new, v_new)
    # only request 1 changed
    pt_np = p.page_table.numpy()
    for kv in (0, 1):
        got_rows = gather_contiguous(pool.reshape(want.shape), pt_np, 2, 1, 200, kv)
        assert np.array_equal(got_rows, gather_contiguous(exp, pt_np, 2, 1, 200, kv))
    changed = pool.reshape(want.shape) != want
    for b in (0, 2):
        for j in range(1):
            for kv in (0, 1):
                assert not changed[pt_np[b, j] * 2 + kv].any(), (b, kv)



# ---------------------------------------------------------------------------
# flat (CSR) page table rebuilt from the lengths

def _flat_golden():
    rows = _rows("flat_page_table.txt")
    g = {"pt": {}, "table": {}, "stale_table": {}}
    for r in rows:
        if r[0] in g:
            g[r[0]][int(r[1])] = [int(v) for v in r[2:]]
        else:
            g[r[0]] = [int(v) for v in r[1:]]
    B = len(g["pt"])
    pt = np.array([g["pt"][b] for b in range(B)], np.int32)
    return g, B, pt


def check_flat_page_table_golden(orc):
    g, B, pt = _flat_golden()
    p = small(lens=g["lens"], T=g["qo_len"][0])
    assert p.max_pages_per_req == g["max_pages"][0]
    x = O.Inputs(p, page_table=torch.from_numpy(pt))
    flat, indptr, bad = orc.flatten_page_table(x)
    n = g["indptr"][-1]
    assert bad == 0
    assert list(indptr) == g["indptr"]
    assert list(flat[:n]) == g["flat"]
    table, bad = orc.page_table_from_flat(x, flat)
    assert bad == 0
    assert table.tolist() == [g["table"][b] for b in range(B)]
    # the correction: restaged from the corrected lengths
    xc = O.Inputs(p, page_table=torch.from_numpy(pt),
                  kv_lens=torch.tensor(g["lens_corrected"], dtype=torch.int32))
    flat_c, indptr_c, _ = orc.flatten_page_table(xc)
    assert list(indptr_c) == g["indptr_corrected"]
    assert list(flat_c[:indptr_c[-1]]) == g["flat_corrected"]
    # the stale flat table read with the corrected lengths misbases rows 2, 3
    stale, _ = orc.page_table_from_flat(xc, flat)
    assert stale.tolist() == [g["stale_table"][b] for b in range(B)]


def check_flat_roundtrip_keeps_verify(orc):
    """flatten -> rebuild returns the used part of the padded table (padding
    -> slot 0), entries past the last row are untouched, and the verify
    output on the rebuilt table is the output on the original."""
    p = small(seed=41, lens=(5, 130, 300, 1, 256), stride=2)
    pt = p.page_table.clone()
    pt[0, 1:] = 7                 # garbage past request 0's used page
    pt[3, :] = 1                  # kv_len 1 < qo_len: invalid, still one page in the layout
    x = O.Inputs(p, page_table=pt)
    sentinel = np.full(p.batch * p.max_pages_per_req, -77, np.int32)
    flat, indptr, bad = orc.flatten_page_table(x, flat_init=sentinel)
    assert bad == 1
    used = [(int(L) + 127) // 128 for L in p.kv_lens]
    assert list(np.diff(indptr)) == used
    assert np.all(flat[indptr[-1]:] == -77)
    table, _ = orc.page_table_from_flat(x, flat)
    ptn = pt.numpy()
    for b, n in enumerate(used):
        assert list(table[b, :n]) == list(ptn[b, :n])
        assert np.all(table[b, n:] == 0)
    o1, _ = orc.verify_dense(x)
    o2, _ = orc.verify_dense(O.Inputs(p, page_table=torch.from_numpy(table)))
    assert np.array_equal(o1, o2)


def check_flat_shrink_across_page_boundary(orc):
    """A length correction across a page boundary: the restaged flat table
    gives the attention of the corrected problem (checked against torch SDPA
    over contiguous K/V read by the numpy layout); the stale one moves the
    later rows onto other pages."""
    T = 2
    p = small(seed=43, lens=(300, 257, 200, 140), T=T, stride=2)
    lens_c = torch.tensor([300, 255, 200, 140], dtype=torch.int32)   # 3 pages -> 2
    xc = O.Inputs(p, kv_lens=lens_c)
    flat_old, _, _ = orc.flatten_page_table(O.Inputs(p))
    flat_new, _, _ = orc.flatten_page_table(xc)
    good, _ = orc.page_table_from_flat(xc, flat_new)
    stale, _ = orc.page_table_from_flat(xc, flat_old)
    out, bad = orc.verify_dense(O.Inputs(p, kv_lens=lens_c, page_table=torch.from_numpy(good)))
    assert bad == 0
    pool5 = pool5_of(p)
    q = q64(p)
    G = p.num_q_heads // p.num_kv_heads
    ptn = p.page_table.numpy()
    for b in range(p.batch):
        L = int(lens_c[b])
        K = decoded(p, gather_contiguous(pool5, ptn, 2, b, L, 0), 0)
        V = decoded(p, gather_contiguous(pool5, ptn, 2, b, L, 1), 1)
        for t in range(T):
            n = L - T + t + 1
            for hq in range(p.num_q_heads):
                want = sdpa(q[b * T + t, hq], K[:n, hq // G], V[:n, hq // G], p.sm_scale)
                assert np.allclose(out[b * T + t, hq], want, atol=1e-12, rtol=1e-12), (b, t, hq)
    assert np.array_equal(stale[:2], good[:2])
    assert not np.array_equal(stale[2:], good[2:])



def check_flat_counts_clamped(orc):
    """Row page counts outside [1, max_pages]: a negative or zero length holds
    no page, a length past the capacity holds max_pages (so later rows keep
    defined bases); the rebuilt table pads with slot 0 either way."""
    p = small(seed=45, lens=(5, 600, 300, 1, 256), max_pages_per_req=3)
    lens = torch.tensor([5, 600, 300, -7, 256], dtype=torch.int32)
    x = O.Inputs(p, kv_lens=lens)
    flat, indptr, bad = orc.flatten_page_table(x)
    assert bad == 2                                     # 600 > 3 * 128, and -7 < qo_len
    assert list(np.diff(indptr)) == [1, 3, 3, 0, 2]
    ptn = p.page_table.numpy()
    assert list(flat[:indptr[-1]]) == [ptn[0, 0], *ptn[1, :3], *ptn[2, :3], *ptn[4, :2]]
    table, _ = orc.page_table_from_flat(x, flat)
    assert table[3].tolist() == [0, 0, 0]
    assert table[4].tolist() == [ptn[4, 0], ptn[4, 1], 0]

# ---------------------------------------------------------------------------
# drafter attention through the P32 sub-page tables

def check_draft_attn_via_view_equals_dense(orc):
    """The P32 tables of the sub-page view address the bytes the P128 table
    does: attention through them equals the dense verify, for T = 1 and a
    ladder, bf16 and FP8, stride 2 and a layer-local stride of 8."""
    for T, dtype, stride in ((1, W.BF16, 2), (3, W.FP8, 8), (1, W.FP8, 8)):
        p = small(seed=47 + T, lens=(33, 130, 300), T=T, stride=stride, kv_dtype=dtype)
        x = O.Inputs(p)
        k_sub, v_sub, _ = orc.subpage_view(x)
        want, bad0 = orc.verify_dense(x)
        got, bad = orc.draft_attn(x, k_sub, v_sub)
        assert bad == bad0 == 0
        assert np.array_equal(got, want), (T, dtype, stride)


def check_draft_attn_shuffled_subpages_vs_sdpa(orc):
    """Decode (qo_len 1) through P32 tables whose sub-pages are an arbitrary
    permutation of the pool's sub-pages (not grouped four to a page): the
    output is SDPA over K/V rows gathered by numpy from the [sub-page, head,
    32, D] view of the pool."""
    p = small(seed=53, lens=(70, 31, 160), T=1, Hq=8, Hk=2, D=32, stride=3)
    nsub_pool = 4 * p.num_slots * p.slot_stride
    nsub = 4 * p.max_pages_per_req
    gen = np.random.default_rng(53)
    k_sub = gen.permutation(nsub_pool)[:p.batch * nsub].reshape(p.batch, nsub).astype(np.int32)
    v_sub = gen.permutation(nsub_pool)[:p.batch * nsub].reshape(p.batch, nsub).astype(np.int32)
    x = O.Inputs(p)
    got, bad = orc.draft_attn(x, k_sub, v_sub)
    assert bad == 0
    subs = pool5_of(p).reshape(nsub_pool, p.num_kv_heads, 32, p.head_dim)
    q = q64(p)
    G = p.num_q_heads // p.num_kv_heads
    for b in range(p.batch):
        L = int(p.kv_lens[b])
        for hq in range(p.num_q_heads):
            h = hq // G
            Kr = np.stack([subs[k_sub[b, i // 32], h, i % 32] for i in range(L)])
            Vr = np.stack([subs[v_sub[b, i // 32], h, i % 32] for i in range(L)])
            want = sdpa(q[b, hq], decoded(p, Kr, 0), decoded(p, Vr, 1), p.sm_scale)
            assert np.allclose(got[b, hq], want, atol=1e-12, rtol=1e-12), (b, hq)


def check_draft_attn_layer_stride_and_invalid(orc):
    """A pool whose slots hold eight buffers (this layer's K and V plus six of
    other layers, here NaN): the view built with the layer-local stride reads
    none of the others.  A used sub-page index outside the view makes the
    request invalid (zero rows); an unused one does not."""
    p = small(seed=59, lens=(40, 129, 250), T=2, stride=8)
    pool = p.pool.clone()
    pool.view(p.num_slots, 8, -1)[:, 2:] = float("nan")
    x = O.Inputs(p, pool=pool)
    k_sub, v_sub, _ = orc.subpage_view(x)
    got, bad = orc.draft_attn(x, k_sub, v_sub)
    assert bad == 0 and np.all(np.isfinite(got))
    want, _ = orc.verify_dense(x)
    assert np.array_equal(got, want)
    limit = 4 * p.num_slots * 8
    k_bad = k_sub.copy()
    k_bad[1, 4] = limit                 # sub-page 4 of request 1 (positions 128..159) is used
    k_bad[0, 5] = limit                 # request 0 uses sub-pages 0..1 only
    got2, bad2 = orc.draft_attn(x, k_bad, v_sub)
    assert bad2 == 1
    T, Hq = p.qo_len, p.num_q_heads
    assert np.all(got2[T:2 * T] == 0)
    assert np.array_equal(got2[:T], got[:T]) and np.array_equal(got2[2 * T:], got[2 * T:])


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
