"""Parity of the flat (CSR) page-table entry points and of the drafter's
attention through the P32 sub-page tables with the fp64 oracle, through the C
ABI.  Tables and indices bit-exact; outputs max-abs 2e-2 (bf16 K/V) or 5e-2
(FP8 K/V) against fp64."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_kv_gb300 as T
from speculative_decode_verify_kv_gb300 import workloads as W
from speculative_decode_verify_kv_gb300.runtime import DeviceVerify

pytestmark = pytest.mark.gpu

TOL_BF16, TOL_FP8 = 2e-2, 5e-2


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


# ---------------------------------------------------------------------------
# flat (CSR) page table

@pytest.mark.parametrize("B,NP", [(5, 3), (600, 5)])   # one CTA; three CTAs of 256 rows
def test_flat_tables_bit_exact(B, NP):
    gen = torch.Generator().manual_seed(B)
    lens = torch.randint(-5, 128 * NP + 40, (B,), generator=gen, dtype=torch.int32)
    lens[:3] = torch.tensor([0, 128, 129], dtype=torch.int32)[:min(3, B)]
    pt = torch.randint(0, 1000, (B, NP), generator=gen, dtype=torch.int32)
    p = W.make_problem(kv_lens=[4] * B, qo_len=4, num_q_heads=2, num_kv_heads=1, head_dim=64,
                       max_pages_per_req=NP, num_slots=1000, seed=1)
    x = oracle.Inputs(p, page_table=pt, kv_lens=lens)
    want_flat, want_indptr, bad = oracle.flatten_page_table(x, flat_init=np.full(B * NP, -77, np.int32))
    g = T.geom_of(p)
    d_pt, d_lens = pt.cuda(), lens.cuda()
    flat = torch.full((B * NP,), -77, dtype=torch.int32, device="cuda")
    indptr = torch.full((B + 1,), -1, dtype=torch.int32, device="cuda")
    T.trtv_get_device_error()
    T.trtv_flatten_page_table(g, d_pt, d_lens, flat, indptr)
    assert np.array_equal(indptr.cpu().numpy(), want_indptr)
    assert np.array_equal(flat.cpu().numpy(), want_flat)
    err = T.trtv_get_device_error()
    assert bool(err & T.DEVERR_KV_LEN) == (bad > 0)
    # and back: the consumer's rebuild from the lengths
    want_pt, _ = oracle.page_table_from_flat(x, want_flat)
    back = torch.full_like(d_pt, -5)
    T.trtv_page_table_from_flat(g, flat, d_lens, back)
    assert np.array_equal(back.cpu().numpy(), want_pt)
    T.trtv_get_device_error()


def test_flat_shrink_across_page_boundary():
    """A length correction moves row 1 from 3 pages to 2.  Restaging the flat
    table from the corrected lengths gives the corrected problem's attention;
    the stale flat table gives what the oracle says it reads (later rows on
    other pages)."""
    p = W.make_problem(kv_lens=[300, 257, 200, 700, 140], qo_len=4, num_q_heads=32, num_kv_heads=4,
                       head_dim=128, seed=61, slack_slots=3)
    dv = DeviceVerify(p, out_dtype="f32")
    stale = dv.flatten()[0].clone()
    lens_c = p.kv_lens.clone()
    lens_c[1] = 255
    dv.kv_lens.copy_(lens_c)
    dv.flatten()
    out = dv.dense_flat().cpu().numpy()
    xc = oracle.Inputs(p, kv_lens=lens_c)
    ref, bad = oracle.verify_dense(xc)
    assert bad == 0
    assert np.abs(out - ref).max() <= TOL_BF16
    # the stale flat table: rows 0 and 1 unchanged, rows 2.. read other pages
    out_stale = dv.dense_flat(flat=stale).cpu().numpy()
    stale_pt, _ = oracle.page_table_from_flat(xc, stale.cpu().numpy())
    ref_stale, _ = oracle.verify_dense(oracle.Inputs(p, kv_lens=lens_c,
                                                     page_table=torch.from_numpy(stale_pt)))
    assert np.abs(out_stale - ref_stale).max() <= TOL_BF16
    assert np.abs(out_stale[8:] - ref[8:]).max() > 0.1
    assert T.trtv_get_device_error() == 0


def test_flat_verify_matches_padded_under_graph_replay():
    """Capture flatten + flat verify once; replays with mutated lengths (a row
    growing and shrinking across page boundaries) match the oracle."""
    p = W.make_problem(kv_lens=[1000, 700, 129, 1500], qo_len=4, num_q_heads=64, num_kv_heads=4,
                       head_dim=128, seed=62, max_pages_per_req=16)
    dv = DeviceVerify(p, out_dtype="f32")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dv.flatten(stream=s)
        dv.dense_flat(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dv.flatten()
        dv.dense_flat()
    for lens in ([1000, 700, 129, 1500], [1024, 513, 128, 1500], [4, 2048, 257, 1]):
        lens_t = torch.tensor(lens, dtype=torch.int32)
        dv.kv_lens.copy_(lens_t)
        graph.replay()
        torch.cuda.synchronize()
        ref, bad = oracle.verify_dense(oracle.Inputs(p, kv_lens=lens_t))
        assert np.abs(dv.out.cpu().numpy() - ref).max() <= TOL_BF16
        err = T.trtv_get_device_error()
        assert bool(err & T.DEVERR_KV_LEN) == (bad > 0)


# ---------------------------------------------------------------------------
# drafter attention through the P32 tables

def _nan_other_layers(p):
    """Buffers 2.. of every slot belong to other layers: fill them with NaN."""
    pool = p.pool.clone()
    if p.kv_dtype == W.FP8:
        pool.view(p.num_slots, p.slot_stride, -1)[:, 2:] = 0x7F      # E4M3 NaN
    else:
        pool.view(p.num_slots, p.slot_stride, -1)[:, 2:] = float("nan")
    return p.with_(pool=pool)


@pytest.mark.parametrize("dtype,Hq,Hk,Tq", [
    (W.BF16, 32, 4, 1),    # drafter decode, 8 rows (mma.sync)
    (W.FP8, 32, 4, 1),     # FP8 draft layer, 8 rows (mma.sync)
    (W.BF16, 64, 4, 4),    # ladder, 64 rows (tcgen05 bf16)
    (W.FP8, 16, 2, 3),     # ladder, 24 -> 32 rows
])
def test_draft_attn_through_view_stride8(dtype, Hq, Hk, Tq):
    """The drafter's view of a pool whose slots hold eight buffers (layer-local
    stride 8; the other six are NaN): the P32 tables from the sub-page view
    give the oracle's attention."""
    p = _nan_other_layers(W.make_problem(kv_lens=[1000, 33, 129, 4096, Tq], qo_len=Tq,
                                         num_q_heads=Hq, num_kv_heads=Hk, head_dim=128,
                                         kv_dtype=dtype, seed=Hq + Tq, slot_stride=8, slack_slots=2))
    dv = DeviceVerify(p, out_dtype="f32")
    k_sub, v_sub = dv.subpage_view()
    out = dv.draft().cpu().numpy()
    x = oracle.Inputs(p)
    ref, bad = oracle.draft_attn(x, k_sub.cpu().numpy(), v_sub.cpu().numpy())
    assert bad == 0
    assert np.all(np.isfinite(out))
    assert np.abs(out - ref).max() <= tol(p)
    assert T.trtv_get_device_error() == 0


@pytest.mark.parametrize("Tq,D", [(1, 128), (3, 64)])
def test_draft_attn_shuffled_subpages(Tq, D):
    """P32 tables whose sub-pages are an arbitrary permutation of the pool's
    sub-pages (not four to a page, any order); unused entries past
    ceil(kv_len / 32) hold out-of-range values and are neither read nor
    flagged."""
    p = W.make_problem(kv_lens=[70, 31, 900, 128], qo_len=Tq, num_q_heads=16, num_kv_heads=2,
                       head_dim=D, seed=63 + Tq, slot_stride=3, slack_slots=4, max_pages_per_req=8)
    nsub_pool = 4 * p.num_slots * p.slot_stride
    nsub = 4 * p.max_pages_per_req
    gen = np.random.default_rng(63)
    k_sub = gen.permutation(nsub_pool)[:p.batch * nsub].reshape(p.batch, nsub).astype(np.int32)
    v_sub = gen.permutation(nsub_pool)[:p.batch * nsub].reshape(p.batch, nsub).astype(np.int32)
    for b, L in enumerate(p.kv_lens.tolist()):
        used = (L + 31) // 32
        k_sub[b, used:] = nsub_pool + 1000
        v_sub[b, used:] = -3
    dv = DeviceVerify(p, out_dtype="f32", num_ctas=7)
    out = dv.draft(torch.from_numpy(k_sub).cuda(), torch.from_numpy(v_sub).cuda()).cpu().numpy()
    ref, bad = oracle.draft_attn(oracle.Inputs(p), k_sub, v_sub)
    assert bad == 0
    assert np.abs(out - ref).max() <= TOL_BF16
    assert T.trtv_get_device_error() == 0


@pytest.mark.parametrize("dtype,Hq", [(W.BF16, 8), (W.FP8, 32)])
def test_draft_attn_bad_subpage_flagged(dtype, Hq):
    p = W.make_problem(kv_lens=[300, 200], qo_len=1, num_q_heads=Hq, num_kv_heads=4 if Hq == 32 else 2,
                       head_dim=128, kv_dtype=dtype, seed=64)
    dv = DeviceVerify(p, out_dtype="f32")
    dv.subpage_view()
    dv.k_sub[1, 2] = 4 * p.num_slots * p.slot_stride     # used by request 1 (positions 64..95)
    out = dv.draft().cpu().numpy()
    assert T.trtv_get_device_error() & T.DEVERR_PAGE_ID
    assert np.all(np.isfinite(out))
    # request 0 is untouched
    x = oracle.Inputs(p)
    k_sub, v_sub, _ = oracle.subpage_view(x)
    ref, _ = oracle.draft_attn(x, k_sub, v_sub)
    assert np.abs(out[:1] - ref[:1]).max() <= tol(p)


def test_draft_attn_bf16_out_and_split_invariance():
    p = W.make_problem(kv_lens=[5000, 1200, 64], qo_len=1, num_q_heads=32, num_kv_heads=4,
                       head_dim=128, seed=65, slot_stride=8)
    x = oracle.Inputs(p)
    k_sub, v_sub, _ = oracle.subpage_view(x)
    ref, _ = oracle.draft_attn(x, k_sub, v_sub)
    for n in (1, 5, 0):
        dv = DeviceVerify(p, out_dtype="bf16", num_ctas=n)
        dv.subpage_view()
        out = dv.draft().float().cpu().numpy()
        assert np.abs(out - ref).max() <= TOL_BF16, n
    assert T.trtv_get_device_error() == 0


def test_draft_attn_graph_replay_with_mutated_lens():
    """Capture the sub-page view and the drafter attention once; replays with
    the lengths grown and shrunk on the device match the oracle on the
    replay's own P32 tables."""
    p = W.make_problem(kv_lens=[700, 2000, 129], qo_len=1, num_q_heads=32, num_kv_heads=4, head_dim=128,
                       kv_dtype=W.FP8, seed=66, slot_stride=8, max_pages_per_req=24)
    dv = DeviceVerify(p, out_dtype="f32")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dv.subpage_view(stream=s)
        dv.draft(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dv.subpage_view()
        dv.draft()
    for lens in ([700, 2000, 129], [3072, 1, 33], [0, 1500, 2048]):
        lens_t = torch.tensor(lens, dtype=torch.int32)
        dv.kv_lens.copy_(lens_t)
        graph.replay()
        torch.cuda.synchronize()
        x = oracle.Inputs(p, kv_lens=lens_t)
        ref, bad = oracle.draft_attn(x, dv.k_sub.cpu().numpy(), dv.v_sub.cpu().numpy())
        assert np.abs(dv.out.cpu().numpy() - ref).max() <= TOL_FP8
        err = T.trtv_get_device_error()
        assert bool(err & T.DEVERR_KV_LEN) == (bad > 0)
