"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerances: max-abs 2e-2 on outputs with bf16 K/V, 5e-2 with FP8 K/V (fp32
accumulation against fp64); proxy scores max-abs 1e-3; sub-page indices and
top-k indices bit-exact (top-k compared on identical scores -- the oracle's
selection run on the GPU's fp32 scores -- and on fresh oracle scores wherever
the k-th boundary gap exceeds 1e-3).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_kv_gb300 as T
from speculative_decode_verify_kv_gb300 import workloads as W
from speculative_decode_verify_kv_gb300.runtime import DeviceVerify

pytestmark = pytest.mark.gpu

TOL_BF16, TOL_FP8, TOL_SCORE = 2e-2, 5e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decode_verify_kv_gb300 import _build
    _build.build()
    T.load()
    T.trtv_get_device_error()  # clear


def tol(p):
    return TOL_FP8 if p.kv_dtype == W.FP8 else TOL_BF16


def sub(p, reqs):
    """The same problem restricted to requests `reqs` (same pool), for the oracle."""
    reqs = list(reqs)
    Tq = p.qo_len
    rows = torch.cat([torch.arange(b * Tq, (b + 1) * Tq) for b in reqs])
    return oracle.Inputs(p, q=p.q[rows], page_table=p.page_table[reqs].contiguous(),
                         kv_lens=p.kv_lens[reqs].contiguous(), batch=len(reqs))


def out_rows(out, p, reqs):
    Tq = p.qo_len
    rows = torch.cat([torch.arange(b * Tq, (b + 1) * Tq) for b in reqs])
    return out.float().cpu()[rows].numpy()


def check_dense(p, num_ctas=0, reqs=None, out_dtype=None):
    dv = DeviceVerify(p, num_ctas=num_ctas, out_dtype=out_dtype)
    out = dv.dense()
    torch.cuda.synchronize()
    reqs = range(p.batch) if reqs is None else reqs
    ref, bad = oracle.verify_dense(sub(p, reqs))
    got = out_rows(out, p, reqs)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    assert err <= tol(p), f"max abs err {err}"
    assert T.trtv_get_device_error() == 0
    return dv, err


# ---------------------------------------------------------------------------
# a1: sub-page view

@pytest.mark.parametrize("stride", [2, 8, 171])
def test_subpage_view_bit_exact(stride):
    p = W.make_problem(kv_lens=[100, 257, 1, 33, 128, 129], qo_len=1, num_q_heads=4, num_kv_heads=2,
                       head_dim=64, slot_stride=stride, seed=stride, slack_slots=3,
                       max_pages_per_req=4)
    dv = DeviceVerify(p)
    k, v = dv.subpage_view()
    rk, rv, bad = oracle.subpage_view(oracle.Inputs(p))
    assert bad == 0
    assert np.array_equal(k.cpu().numpy(), rk) and np.array_equal(v.cpu().numpy(), rv)
    assert T.trtv_get_device_error() == 0


# ---------------------------------------------------------------------------
# a2 + a6: dense ladder verify with split-KV combine

def test_dense_tiny_workload():
    p = W.make_workload("tiny")
    check_dense(p)


@pytest.mark.parametrize("num_ctas", [1, 3, 7, 64, 300])
def test_dense_split_invariance(num_ctas):
    p = W.make_problem(kv_lens=[1000, 37, 513, 4, 2000], qo_len=4, num_q_heads=32, num_kv_heads=4,
                       head_dim=128, seed=11, slack_slots=5)
    dv1, e1 = check_dense(p, num_ctas=num_ctas, out_dtype="f32")
    dv2 = DeviceVerify(p, num_ctas=1, out_dtype="f32")
    o2 = dv2.dense()
    torch.cuda.synchronize()
    # a split changes the running maximum that P is rounded against before the
    # bf16 PV product, so splits agree to bf16 rounding of P, not fp32 rounding
    assert (dv1.out - o2).abs().max().item() < 5e-3


@pytest.mark.parametrize("num_ctas", [40, 100, 1024])
def test_dense_one_sequence_over_many_ctas(num_ctas):
    """One (request, KV head) sequence of 63 pages cut among up to 40 CTAs (more
    contributors than a warp has lanes), or among 100 / 1024 CTAs of which
    most get no page (empty ranges leave no partial)."""
    p = W.make_problem(kv_lens=[8000], qo_len=4, num_q_heads=8, num_kv_heads=1, head_dim=128,
                       seed=13, slack_slots=2)
    check_dense(p, num_ctas=num_ctas, out_dtype="f32")


def test_workspace_needs_no_initial_contents():
    """A workspace full of 0xFF bytes (NaN partials, -1 descriptors) gives the
    same results: every call writes what it reads."""
    p = W.make_problem(kv_lens=[1000, 37, 513, 4, 2000], qo_len=4, num_q_heads=64, num_kv_heads=4,
                       head_dim=128, seed=17, slack_slots=5, topk=4, max_pages_per_req=16)
    dv = DeviceVerify(p, num_ctas=9, out_dtype="f32")
    dv.workspace.fill_(255)
    out = dv.dense().cpu().numpy()
    ref, _ = oracle.verify_dense(oracle.Inputs(p))
    assert np.abs(out - ref).max() <= TOL_BF16
    dv.workspace.fill_(255)
    dv.proxy()
    idx = dv.select()
    dv.workspace.fill_(255)
    sp = dv.sparse().cpu().numpy()
    ref, bad = oracle.sparse_attn(oracle.Inputs(p), idx.cpu().numpy())
    assert bad == 0
    assert np.abs(sp - ref).max() <= TOL_BF16
    assert T.trtv_get_device_error() == 0


@pytest.mark.parametrize("Hq,Hk,Tq,D", [
    (8, 8, 4, 128),    # G = 1
    (16, 1, 4, 128),   # G = 16, 64 rows
    (64, 4, 8, 128),   # G = 16, T = 8, 128 rows
    (12, 2, 4, 128),   # G = 6 padded to 8
    (64, 2, 2, 128),   # G = 32 > 16
    (8, 2, 1, 64),     # decode, D = 64
    (32, 4, 4, 64),
    (4, 4, 16, 128),   # long draft
])
def test_dense_shapes(Hq, Hk, Tq, D):
    p = W.make_problem(kv_lens=[300, 129, 1000, Tq, 256], qo_len=Tq, num_q_heads=Hq,
                       num_kv_heads=Hk, head_dim=D, seed=Hq * 7 + Tq, slack_slots=4, slot_stride=3)
    check_dense(p, num_ctas=5, out_dtype="f32")
    check_dense(p, out_dtype="bf16")


def test_dense_qo_len_1_is_decode():
    p = W.make_problem(kv_lens=[77, 1024, 3000], qo_len=1, num_q_heads=32, num_kv_heads=4,
                       head_dim=128, seed=5)
    check_dense(p, out_dtype="f32")


@pytest.mark.parametrize("Hq,Hk", [(8, 2), (32, 2)])  # 16 rows (mma.sync), 64 rows (tcgen05)
def test_dense_stale_pages_hold_nan(Hq, Hk):
    """Positions past kv_len inside a page and unused slots hold NaN: the
    output must not see them."""
    p = W.make_problem(kv_lens=[100, 257, 130], qo_len=4, num_q_heads=Hq, num_kv_heads=Hk,
                       head_dim=128, seed=9, slack_slots=3, fill_unused_with=float("nan"))
    pool = p.pool.clone()
    x = oracle.Inputs(p)
    # poison every element of the used pages that lies past its request's length
    flat = pool.view(-1)
    for b in range(p.batch):
        L = int(p.kv_lens[b])
        for pos in range(L, ((L + 127) // 128) * 128):
            for h in range(p.num_kv_heads):
                for kv in (0, 1):
                    off = oracle.element_offset(int(p.page_table[b, pos // 128]), p.slot_stride,
                                                p.num_kv_heads, p.head_dim, pos, h, kv, 0)
                    flat[off:off + p.head_dim] = float("nan")
    p2 = p.with_(pool=pool)
    check_dense(p2, out_dtype="f32")
    check_dense(p2, num_ctas=2, out_dtype="f32")


@pytest.mark.parametrize("Hq,Hk", [(32, 4), (64, 4)])
def test_dense_fp8_stale_positions_hold_nan(Hq, Hk):
    """FP8 cache: positions past kv_len inside used pages hold the E4M3 NaN
    code (0x7F); the output must not see them."""
    p = W.make_problem(kv_lens=[100, 257, 130, 4], qo_len=4, num_q_heads=Hq, num_kv_heads=Hk,
                       head_dim=128, kv_dtype=W.FP8, seed=19, slack_slots=3)
    pool = p.pool.clone()
    flat = pool.view(torch.uint8).view(-1)
    for b in range(p.batch):
        L = int(p.kv_lens[b])
        for pos in range(L, ((L + 127) // 128) * 128):
            for h in range(p.num_kv_heads):
                for kv in (0, 1):
                    off = oracle.element_offset(int(p.page_table[b, pos // 128]), p.slot_stride,
                                                p.num_kv_heads, p.head_dim, pos, h, kv, 0)
                    flat[off:off + p.head_dim] = 0x7F
    p2 = p.with_(pool=pool)
    check_dense(p2, out_dtype="f32")
    check_dense(p2, num_ctas=5, out_dtype="f32")


def test_dense_fp8():
    p = W.make_problem(kv_lens=[4096, 300, 129, 1000, 77, 2500], qo_len=4, num_q_heads=32,
                       num_kv_heads=4, head_dim=128, kv_dtype=W.FP8, seed=21, slack_slots=3)
    check_dense(p, out_dtype="f32")
    check_dense(p, num_ctas=9, out_dtype="bf16")
    # independent K and V scales
    check_dense(p.with_(k_scale=p.k_scale * 0.5, v_scale=p.v_scale * 3.0), out_dtype="f32")


def test_dense_fp8_shapes():
    for Hq, Hk, Tq in ((8, 8, 4), (64, 4, 8), (16, 1, 4), (32, 4, 1)):
        p = W.make_problem(kv_lens=[300, 129, Tq, 1000], qo_len=Tq, num_q_heads=Hq, num_kv_heads=Hk,
                           head_dim=128, kv_dtype=W.FP8, seed=Hq + Tq, slack_slots=2)
        check_dense(p, num_ctas=3, out_dtype="f32")


def test_dense_edge_lengths():
    # kv_len == qo_len, page-aligned, full capacity
    p = W.make_problem(kv_lens=[4, 128, 256, 512, 32, 33], qo_len=4, num_q_heads=16, num_kv_heads=2,
                       head_dim=128, seed=3, max_pages_per_req=4, slack_slots=2)
    check_dense(p, out_dtype="f32")
    check_dense(p, num_ctas=11, out_dtype="f32")


@pytest.mark.parametrize("D", [64, 128])
def test_dense_invalid_requests_are_zero_and_flagged(D):
    p = W.make_problem(kv_lens=[300, 200, 100], qo_len=4, num_q_heads=8, num_kv_heads=2,
                       head_dim=D, seed=4, max_pages_per_req=3)
    lens = p.kv_lens.clone()
    lens[1] = 2           # shorter than qo_len
    lens[2] = 1000        # beyond capacity (3 pages)
    dv = DeviceVerify(p, out_dtype="f32")
    dv.kv_lens.copy_(lens)
    out = dv.dense().cpu()
    err = T.trtv_get_device_error()
    assert err & T.DEVERR_KV_LEN
    assert torch.all(out[4:12] == 0)
    out = out.reshape(12, 8, D)
    ref, bad = oracle.verify_dense(oracle.Inputs(p, kv_lens=lens))
    assert bad == 2
    assert np.abs(out.numpy() - ref).max() <= TOL_BF16
    assert T.trtv_get_device_error() == 0


def test_dense_bad_page_id_flagged():
    p = W.make_problem(kv_lens=[300, 200], qo_len=4, num_q_heads=8, num_kv_heads=2, head_dim=64,
                       seed=6)
    dv = DeviceVerify(p, out_dtype="f32")
    dv.page_table[1, 0] = p.num_slots + 5
    dv.dense()
    assert T.trtv_get_device_error() & T.DEVERR_PAGE_ID


@pytest.mark.parametrize("Hq,Hk", [(32, 4), (64, 4), (16, 2)])   # tcgen05 E4M3: 32 / 64 / 32 rows
def test_dense_fp8_invalid_requests_and_bad_page(Hq, Hk):
    """FP8 caches on the tensor-core path: invalid kv_len rows are zero and
    flagged, a bad page id is flagged, and the valid requests still match."""
    p = W.make_problem(kv_lens=[300, 200, 100, 700], qo_len=4, num_q_heads=Hq, num_kv_heads=Hk,
                       head_dim=128, kv_dtype=W.FP8, seed=8, max_pages_per_req=6)
    lens = p.kv_lens.clone()
    lens[1] = 2           # shorter than qo_len
    lens[2] = 1000        # beyond capacity (6 pages)
    dv = DeviceVerify(p, num_ctas=7, out_dtype="f32")
    dv.kv_lens.copy_(lens)
    out = dv.dense().cpu()
    assert T.trtv_get_device_error() & T.DEVERR_KV_LEN
    assert torch.all(out[4:12] == 0)
    ref, bad = oracle.verify_dense(oracle.Inputs(p, kv_lens=lens))
    assert bad == 2
    assert np.abs(out.numpy() - ref).max() <= TOL_FP8
    dv.kv_lens.copy_(p.kv_lens)
    dv.page_table[3, 1] = p.num_slots + 5
    dv.dense()
    assert T.trtv_get_device_error() & T.DEVERR_PAGE_ID


def test_sparse_fp8_full_k_equals_dense():
    """k >= valid blocks on an FP8 cache: the sparse pass equals the dense one
    (both on the tensor-core E4M3 path, 64 rows)."""
    p = W.make_problem(kv_lens=[1000, 129, 4, 700], qo_len=4, num_q_heads=64, num_kv_heads=4,
                       head_dim=128, kv_dtype=W.FP8, seed=44, topk=8, max_pages_per_req=8)
    dv = DeviceVerify(p, out_dtype="f32")
    dense = dv.dense().clone()
    dv.proxy()
    dv.select()
    sp = dv.sparse()
    torch.cuda.synchronize()
    assert (dense - sp).abs().max().item() < 2e-2
    ref, _ = oracle.verify_dense(oracle.Inputs(p))
    assert np.abs(sp.cpu().numpy() - ref).max() <= TOL_FP8


@pytest.mark.parametrize("Hq", [32, 64])  # 32 rows (mma.sync), 64 rows (tcgen05)
def test_dense_graph_replay_with_mutated_lens(Hq):
    """Capture once, then grow and shrink kv_lens on the device between replays
    (including beyond the first call's maximum): every replay matches."""
    p = W.make_problem(kv_lens=[200, 900, 50, 1400], qo_len=4, num_q_heads=Hq, num_kv_heads=4,
                       head_dim=128, seed=8, max_pages_per_req=16, slack_slots=40)
    full = W.make_problem(kv_lens=[2048, 2048, 2048, 2048], qo_len=4, num_q_heads=Hq, num_kv_heads=4,
                          head_dim=128, seed=8, max_pages_per_req=16)
    dv = DeviceVerify(full, out_dtype="f32")
    s = torch.cuda.Stream()
    dv.kv_lens.copy_(p.kv_lens)
    with torch.cuda.stream(s):
        dv.dense(stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dv.dense(stream=s)
    for lens in ([200, 900, 50, 1400], [2048, 5, 1300, 1401], [4, 4, 2047, 700], [2048] * 4):
        lt = torch.tensor(lens, dtype=torch.int32)
        dv.kv_lens.copy_(lt)
        g.replay()
        torch.cuda.synchronize()
        ref, bad = oracle.verify_dense(oracle.Inputs(full, kv_lens=lt))
        assert np.abs(dv.out.cpu().numpy() - ref).max() <= TOL_BF16, lens
    assert T.trtv_get_device_error() == 0


# ---------------------------------------------------------------------------
# a3 proxy, a4 top-k, a5 sparse

def check_proxy(p, num_ctas=0, reqs=None):
    dv = DeviceVerify(p, num_ctas=num_ctas)
    sc = dv.proxy().cpu().numpy()
    reqs = list(range(p.batch)) if reqs is None else list(reqs)
    ref, bad = oracle.proxy_score(sub(p, reqs))
    got = sc[reqs]
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    f = np.isfinite(ref)
    err = np.abs(got[f] - ref[f]).max()
    assert err <= TOL_SCORE, err
    assert T.trtv_get_device_error() == 0
    return dv, sc


@pytest.mark.parametrize("Hq,Hk,Tq,dt", [
    (64, 4, 4, W.BF16), (64, 4, 8, W.BF16), (8, 2, 4, W.BF16), (8, 8, 1, W.BF16),
    (12, 2, 4, W.BF16), (64, 4, 4, W.FP8), (16, 4, 3, W.FP8),
])
def test_proxy_scores(Hq, Hk, Tq, dt):
    p = W.make_problem(kv_lens=[1000, 129, Tq, 3000, 256], qo_len=Tq, num_q_heads=Hq, num_kv_heads=Hk,
                       head_dim=128, kv_dtype=dt, seed=Hq + 3 * Tq, slack_slots=3, max_pages_per_req=30)
    check_proxy(p)
    check_proxy(p, num_ctas=4)


def test_topk_bit_exact_on_gpu_scores():
    p = W.make_problem(kv_lens=[5000, 129, 4, 20000, 1024, 777], qo_len=4, num_q_heads=64,
                       num_kv_heads=4, head_dim=128, seed=31, topk=16, max_pages_per_req=160)
    dv, sc = check_proxy(p)
    for k in (1, 7, 16, 100, 160):
        dv.topk = k
        dv.block_idx = torch.empty(p.batch, p.qo_len, p.num_kv_heads, k, dtype=torch.int32, device="cuda")
        got = dv.select().cpu().numpy()
        ref, bad = oracle.topk(oracle.Inputs(p), sc.astype(np.float64), k)
        assert np.array_equal(got, ref), k


def test_topk_ties_and_negative_zero():
    p = W.make_problem(kv_lens=[128 * 40, 128 * 7 + 3], qo_len=4, num_q_heads=8, num_kv_heads=2,
                       head_dim=64, seed=2, topk=5, max_pages_per_req=40)
    dv = DeviceVerify(p)
    rng = np.random.default_rng(0)
    s = rng.integers(-2, 3, size=(p.batch, 4, 2, 40)).astype(np.float32)
    s[s == 0] = -0.0
    s[0, 0, 0, ::2] = 0.0
    sc = torch.from_numpy(s).cuda()
    got = dv.select(scores=sc).cpu().numpy()
    ref, _ = oracle.topk(oracle.Inputs(p), s.astype(np.float64), 5)
    assert np.array_equal(got, ref)


def test_topk_fresh_scores_where_gap_is_clear():
    p = W.make_workload("msa", batch=4)
    dv = DeviceVerify(p)
    dv.proxy()
    got = dv.select().cpu().numpy()
    x = oracle.Inputs(p)
    s64, _ = oracle.proxy_score(x)
    ref, _ = oracle.topk(x, s64, p.topk)
    checked = 0
    for b in range(p.batch):
        for t in range(p.qo_len):
            for h in range(p.num_kv_heads):
                n = (int(p.kv_lens[b]) - p.qo_len + t) // 128 + 1
                srt = np.sort(s64[b, t, h, :n])[::-1]
                if n > p.topk and srt[p.topk - 1] - srt[p.topk] <= 1e-3:
                    continue
                assert np.array_equal(got[b, t, h], ref[b, t, h])
                checked += 1
    assert checked >= 0.9 * p.batch * p.qo_len * p.num_kv_heads


@pytest.mark.parametrize("num_ctas", [0, 5])
def test_sparse_with_identical_indices(num_ctas):
    p = W.make_problem(kv_lens=[5000, 129, 4, 3000, 1024], qo_len=4, num_q_heads=64, num_kv_heads=4,
                       head_dim=128, seed=41, topk=8, max_pages_per_req=40)
    dv = DeviceVerify(p, num_ctas=num_ctas, out_dtype="f32")
    dv.proxy()
    idx = dv.select()
    out = dv.sparse().cpu().numpy()
    ref, bad = oracle.sparse_attn(oracle.Inputs(p), idx.cpu().numpy())
    assert bad == 0
    assert np.abs(out - ref).max() <= TOL_BF16
    assert T.trtv_get_device_error() == 0


def test_sparse_full_k_equals_dense():
    p = W.make_problem(kv_lens=[1000, 129, 4, 700], qo_len=4, num_q_heads=32, num_kv_heads=4,
                       head_dim=128, seed=43, topk=8, max_pages_per_req=8)
    dv = DeviceVerify(p, out_dtype="f32")
    dense = dv.dense().clone()
    dv.proxy()
    dv.select()
    sp = dv.sparse()
    torch.cuda.synchronize()
    assert (dense - sp).abs().max().item() < 5e-3


def test_sparse_handmade_indices():
    """Duplicates, -1 padding, blocks past a token's bound or past kv_len, and an
    out-of-range index (that token's rows are zero and the error bit is set)."""
    p = W.make_problem(kv_lens=[1000, 300], qo_len=4, num_q_heads=16, num_kv_heads=2,
                       head_dim=128, seed=45, topk=4, max_pages_per_req=10)
    dv = DeviceVerify(p, out_dtype="f32")
    idx = torch.full((2, 4, 2, 4), -1, dtype=torch.int32)
    idx[0, :, :, 0] = 7
    idx[0, :, :, 1] = 7
    idx[0, 1, :, 2] = 2
    idx[0, 2, 0, 3] = 9       # past kv_len (8 pages)
    idx[1, :, :, 0] = 2       # last page of request 1 (positions 256..299)
    idx[1, 3, 1, 1] = 0
    idx[1, 0, 0, 2] = 12      # >= max_pages: token 0 of request 1, head 0 attends nothing
    out = dv.sparse(block_idx=idx.cuda()).cpu().numpy()
    assert T.trtv_get_device_error() & T.DEVERR_BLOCK_IDX
    ref, bad = oracle.sparse_attn(oracle.Inputs(p), idx.numpy())
    assert bad == 1
    assert np.abs(out - ref).max() <= TOL_BF16


def test_msa_pipeline_fp8():
    p = W.make_problem(kv_lens=[6000, 129, 2000], qo_len=4, num_q_heads=64, num_kv_heads=4,
                       head_dim=128, kv_dtype=W.FP8, seed=47, topk=8, slack_slots=3)
    dv = DeviceVerify(p, out_dtype="f32")
    out = dv.msa().cpu().numpy()
    idx = dv.block_idx.cpu().numpy()
    x = oracle.Inputs(p)
    ref, bad = oracle.sparse_attn(x, idx)
    assert np.abs(out - ref).max() <= TOL_FP8
    ref_idx, _ = oracle.topk(x, dv.scores.cpu().numpy().astype(np.float64), p.topk)
    assert np.array_equal(idx, ref_idx)


@pytest.mark.parametrize("Hq,Hk,Tq,num_ctas", [(32, 4, 4, 0), (32, 4, 4, 7), (16, 4, 4, 3), (8, 8, 2, 0)])
def test_sparse_fp8_small_tiles(Hq, Hk, Tq, num_ctas):
    """FP8 sparse attention on tiles of at most 32 rows (the position-major
    tensor-core kernel: 32, 16 and 2 rows), on the GPU's own selection and on
    the full selection (= dense)."""
    p = W.make_problem(kv_lens=[3000, 129, Tq, 1500, 700], qo_len=Tq, num_q_heads=Hq, num_kv_heads=Hk,
                       head_dim=128, kv_dtype=W.FP8, seed=Hq + Tq + num_ctas, topk=6, max_pages_per_req=24,
                       slack_slots=3)
    dv = DeviceVerify(p, num_ctas=num_ctas, out_dtype="f32")
    out = dv.msa().cpu().numpy()
    idx = dv.block_idx.cpu().numpy()
    x = oracle.Inputs(p)
    ref, bad = oracle.sparse_attn(x, idx)
    assert bad == 0
    assert np.abs(out - ref).max() <= TOL_FP8
    npg = torch.tensor([(int(L) + 127) // 128 for L in p.kv_lens])
    full = torch.arange(24, dtype=torch.int32).view(1, 1, 1, 24).expand(p.batch, Tq, Hk, 24)
    full = torch.where(full < npg.view(-1, 1, 1, 1), full, torch.full_like(full, -1)).contiguous()
    dv24 = DeviceVerify(p, num_ctas=num_ctas, out_dtype="f32", topk=24)  # workspace for 24-block lists
    out2 = dv24.sparse(block_idx=full.cuda(), topk=24).cpu().numpy()
    dense_ref, _ = oracle.verify_dense(x)
    assert np.abs(out2 - dense_ref).max() <= TOL_FP8
    assert T.trtv_get_device_error() == 0


def test_fp8_graph_replay_with_mutated_lens():
    """FP8 cache, 32-row tiles: capture once, replay with kv_lens changed on the device."""
    full = W.make_problem(kv_lens=[2048, 2048, 2048, 2048], qo_len=4, num_q_heads=32, num_kv_heads=4,
                          head_dim=128, kv_dtype=W.FP8, seed=88, max_pages_per_req=16)
    dv = DeviceVerify(full, out_dtype="f32")
    s = torch.cuda.Stream()
    dv.kv_lens.copy_(torch.tensor([200, 900, 50, 1400], dtype=torch.int32))
    with torch.cuda.stream(s):
        dv.dense(stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dv.dense(stream=s)
    for lens in ([200, 900, 50, 1400], [2048, 5, 1300, 1401], [4, 4, 2047, 700]):
        lt = torch.tensor(lens, dtype=torch.int32)
        dv.kv_lens.copy_(lt)
        g.replay()
        torch.cuda.synchronize()
        ref, _ = oracle.verify_dense(oracle.Inputs(full, kv_lens=lt))
        assert np.abs(dv.out.cpu().numpy() - ref).max() <= TOL_FP8, lens
    assert T.trtv_get_device_error() == 0


# ---------------------------------------------------------------------------
# KV slot staging along the ladder (bit-exact against the oracle)

@pytest.mark.parametrize("dtype,stride,D", [(W.BF16, 2, 128), (W.BF16, 8, 64), (W.FP8, 2, 128), (W.FP8, 5, 128)])
def test_stage_kv_bit_exact(dtype, stride, D):
    Tq, Hk = 4, 4
    p = W.make_problem(kv_lens=[1000, 4, 127, 128, 129, 3, 600], qo_len=Tq, num_q_heads=4 * Hk, num_kv_heads=Hk,
                       head_dim=D, slot_stride=stride, kv_dtype=dtype, seed=51 + stride, slack_slots=3,
                       max_pages_per_req=8)
    if dtype == W.FP8:
        p = p.with_(k_scale=0.013, v_scale=0.021)
    pt = p.page_table.clone()
    pt[6, 4] = p.num_slots + 9            # request 6: its staged page names no slot
    p = p.with_(page_table=pt)
    g = torch.Generator().manual_seed(7)
    k_new = (torch.randn(p.batch * Tq, Hk, D, generator=g) * 3).to(torch.bfloat16)
    v_new = (torch.randn(p.batch * Tq, Hk, D, generator=g) * 3).to(torch.bfloat16)
    k_new[0, 0, :4] = torch.tensor([1e4, -1e4, float("nan"), 0.0])   # saturation, NaN, zero
    want, bad = oracle.stage_kv(oracle.Inputs(p), k_new, v_new)
    assert bad == 2                       # request 5 (kv_len 3 < qo_len) and request 6
    dv = DeviceVerify(p)
    dv.stage(k_new.cuda(), v_new.cuda())
    torch.cuda.synchronize()
    got = dv.pool.cpu()
    got = got.view(torch.uint8) if dtype == W.FP8 else got.view(torch.int16)
    assert np.array_equal(got.numpy().reshape(-1).view(want.dtype), want.reshape(-1)), "pool differs"
    err = T.trtv_get_device_error()
    assert err & T.DEVERR_KV_LEN and err & T.DEVERR_PAGE_ID


def test_stage_kv_then_verify_reads_the_new_tokens():
    """Staging followed by the dense verify equals the oracle's verify over the
    staged pool (the ladder rows see exactly the new keys and values)."""
    p = W.make_problem(kv_lens=[700, 129, 4000], qo_len=4, num_q_heads=32, num_kv_heads=4, head_dim=128,
                       seed=57, slack_slots=2)
    g = torch.Generator().manual_seed(8)
    k_new = torch.randn(p.batch * 4, 4, 128, generator=g).to(torch.bfloat16)
    v_new = torch.randn(p.batch * 4, 4, 128, generator=g).to(torch.bfloat16)
    pool, bad = oracle.stage_kv(oracle.Inputs(p), k_new, v_new)
    assert bad == 0
    dv = DeviceVerify(p, out_dtype="f32")
    dv.stage(k_new.cuda(), v_new.cuda())
    out = dv.dense().cpu().numpy()
    staged = torch.from_numpy(pool.view(np.int16)).view(torch.bfloat16).reshape(p.pool.shape)
    ref, _ = oracle.verify_dense(oracle.Inputs(p, pool=staged))
    assert np.abs(out - ref).max() <= TOL_BF16
    assert T.trtv_get_device_error() == 0
