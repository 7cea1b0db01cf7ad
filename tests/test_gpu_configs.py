"""Parity with the fp64 oracle at the five verify configurations' own shapes,
run through the C ABI on the production launch (default grid: one CTA per
SM, so the stream-K cut is the one the benchmark times).

The GPU always runs the whole workload; the oracle checks every request where
it finishes in seconds (dense, drafter) and a stated subset elsewhere (the
longest and shortest rows of the FP8 length mix, the first requests of the
MSA and long-context workloads).  Tolerances are the parity suite's: max-abs
2e-2 (bf16 K/V) and 5e-2 (FP8 K/V) on outputs, 1e-3 on proxy scores, top-k
bit-exact on the GPU's own scores and on fresh oracle scores wherever the
k-th boundary gap exceeds 1e-3.

Sources of the definitions checked: "Eagle3 for M3 MSA path + CUDA graphs
compatibility" (fork PR #3), verify commit (ladder, proxy pass, top-k limited
to each token's valid pages, sparse GQA attention over the selected blocks).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_kv_gb300 as T
from speculative_decode_verify_kv_gb300 import workloads as W
from speculative_decode_verify_kv_gb300.runtime import DeviceVerify

pytestmark = pytest.mark.gpu

TOL_BF16, TOL_FP8, TOL_SCORE, GAP = 2e-2, 5e-2, 1e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decode_verify_kv_gb300 import _build
    _build.build()
    T.load()
    T.trtv_get_device_error()  # clear


_WL = {}


def workload(name):
    if name not in _WL:
        _WL.clear()   # one full-size workload on the host at a time
        _WL[name] = W.make_workload(name)
    return _WL[name]


def sub(p, reqs):
    """Oracle inputs for requests `reqs` of problem p (same pool)."""
    reqs = list(reqs)
    rows = torch.cat([torch.arange(b * p.qo_len, (b + 1) * p.qo_len) for b in reqs])
    return oracle.Inputs(p, q=p.q[rows], page_table=p.page_table[reqs].contiguous(),
                         kv_lens=p.kv_lens[reqs].contiguous(), batch=len(reqs))


def rows_of(out, p, reqs):
    rows = torch.cat([torch.arange(b * p.qo_len, (b + 1) * p.qo_len) for b in reqs])
    return out.float().cpu()[rows].numpy()


def tol(p):
    return TOL_FP8 if p.kv_dtype == W.FP8 else TOL_BF16


def check_msa(p, dv, reqs):
    """Proxy scores, top-k and sparse attention of workload p on the GPU (the
    whole batch) against the oracle on requests `reqs`."""
    scores = dv.proxy().clone()
    idx = dv.select().clone()
    out = dv.sparse().clone()
    torch.cuda.synchronize()
    assert T.trtv_get_device_error() == 0
    sc = scores.cpu().numpy()
    gi = idx.cpu().numpy()
    # top-k bit-exact on the GPU's own scores, every request
    ref_i, bad = oracle.topk(oracle.Inputs(p), sc.astype(np.float64), p.topk)
    assert bad == 0
    assert np.array_equal(gi, ref_i)
    # proxy scores on the sampled requests
    x = sub(p, reqs)
    s64, bad = oracle.proxy_score(x)
    assert bad == 0
    got = sc[reqs]
    assert np.array_equal(np.isneginf(got), np.isneginf(s64))
    f = np.isfinite(s64)
    assert np.abs(got[f] - s64[f]).max() <= TOL_SCORE
    # top-k on fresh oracle scores wherever the k-th boundary gap is clear
    fresh, _ = oracle.topk(x, s64, p.topk)
    checked = total = 0
    for i, b in enumerate(reqs):
        for t in range(p.qo_len):
            for h in range(p.num_kv_heads):
                total += 1
                n = (int(p.kv_lens[b]) - p.qo_len + t) // 128 + 1
                srt = np.sort(s64[i, t, h, :n])[::-1]
                if n > p.topk and srt[p.topk - 1] - srt[p.topk] <= GAP:
                    continue
                assert np.array_equal(gi[b, t, h], fresh[i, t, h]), (b, t, h)
                checked += 1
    assert checked >= 0.5 * total
    # sparse attention on the GPU's indices
    ref_o, bad = oracle.sparse_attn(x, gi[reqs])
    assert bad == 0
    err = np.abs(rows_of(out, p, reqs) - ref_o).max()
    assert err <= tol(p), err
    return idx, out


def test_config_dense_full_batch():
    """Dense Eagle3 draft-layer verify: batch 64, qo_len 4, kv_len U{1024..8192},
    32/4 heads, bf16, 12k-slot pool; all 64 requests against the oracle."""
    p = workload("dense")
    dv = DeviceVerify(p)
    k, v = dv.subpage_view()
    out = dv.dense()
    torch.cuda.synchronize()
    rk, rv, bad = oracle.subpage_view(oracle.Inputs(p))
    assert bad == 0
    assert np.array_equal(k.cpu().numpy(), rk) and np.array_equal(v.cpu().numpy(), rv)
    ref, bad = oracle.verify_dense(oracle.Inputs(p))
    assert bad == 0
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    assert err <= TOL_BF16, err
    assert T.trtv_get_device_error() == 0


def test_config_fp8_length_mix():
    """FP8 decode-shaped verify: batch 256, kv_len lognormal clipped to
    [256, 32768], E4M3 K/V; the GPU runs the whole batch, the oracle checks the
    eight longest rows (the clip at 32768 included) and the eight shortest."""
    p = workload("fp8")
    lens = p.kv_lens.numpy()
    order = np.argsort(lens, kind="stable")
    reqs = sorted(set(order[:8].tolist()) | set(order[-8:].tolist()))
    assert lens.max() == 32768 and lens[reqs].max() == 32768 and lens[reqs].min() == lens.min()
    dv = DeviceVerify(p)
    out = dv.dense()
    torch.cuda.synchronize()
    assert T.trtv_get_device_error() == 0
    ref, bad = oracle.verify_dense(sub(p, reqs))
    assert bad == 0
    got = rows_of(out, p, reqs)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    assert err <= TOL_FP8, err


def test_config_msa():
    """MSA sparse verify: batch 32, kv_len U{16384..65536}, 64/4 heads, top-k 16;
    the GPU runs all 32 requests, the oracle checks the first 8 (and the
    top-k of all 32 on the GPU's scores)."""
    p = workload("msa")
    dv = DeviceVerify(p)
    idx, out = check_msa(p, dv, list(range(8)))
    # the fused select returns the same indices at this shape
    dv.block_idx.fill_(-7)
    dv.select_fused()
    torch.cuda.synchronize()
    assert torch.equal(dv.block_idx, idx)
    assert T.trtv_get_device_error() == 0


def test_config_long_context_msa():
    """Long-context MSA verify: batch 8, qo_len 8 (128-row tiles), kv_len
    131072, 64/4 heads, 5 % of K pages shifted by +2.0, top-k 32; the oracle
    checks request 0's scores, selections and sparse output."""
    p = workload("long")
    dv = DeviceVerify(p)
    check_msa(p, dv, [0])


def test_config_drafter_p32():
    """The drafter's FP8 decode step through the P32 tables (slot stride 8,
    other layers' buffers in the slot), the whole batch against the oracle."""
    p = workload("draft")
    dv = DeviceVerify(p)
    k, v = dv.subpage_view()
    out = dv.draft()
    torch.cuda.synchronize()
    assert T.trtv_get_device_error() == 0
    ref, bad = oracle.draft_attn(oracle.Inputs(p), k.cpu().numpy(), v.cpu().numpy())
    assert bad == 0
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= TOL_FP8, err


@pytest.mark.parametrize("num_ctas", [0, 5])
def test_sparse_128_row_tiles(num_ctas):
    """The long-context tile at a small size: 64/4 heads, qo_len 8 (G * T = 128
    rows, 8-token block masks), top-k 32 over lengths that cross page
    boundaries; sparse output on identical indices and on the fused select."""
    p = W.make_problem(kv_lens=[5000, 129, 8, 4100, 1023, 16384], qo_len=8, num_q_heads=64,
                       num_kv_heads=4, head_dim=128, seed=61 + num_ctas, topk=32,
                       max_pages_per_req=128, slack_slots=5)
    dv = DeviceVerify(p, num_ctas=num_ctas, out_dtype="f32")
    dv.proxy()
    idx = dv.select().clone()
    out = dv.sparse().cpu().numpy()
    x = oracle.Inputs(p)
    ref, bad = oracle.sparse_attn(x, idx.cpu().numpy())
    assert bad == 0
    assert np.abs(out - ref).max() <= TOL_BF16
    ref_i, _ = oracle.topk(x, dv.scores.cpu().double().numpy(), p.topk)
    assert np.array_equal(idx.cpu().numpy(), ref_i)
    dv.block_idx.fill_(-7)
    dv.select_fused()
    torch.cuda.synchronize()
    assert torch.equal(dv.block_idx, idx)
    out2 = dv.sparse().cpu().numpy()
    assert np.abs(out2 - ref).max() <= TOL_BF16
    # k >= every token's valid pages: the sparse pass is the dense one
    dense_ref, _ = oracle.verify_dense(x)
    full = torch.arange(128, dtype=torch.int32).view(1, 1, 1, 128).expand(p.batch, 8, 4, 128)
    full = torch.where(full < torch.tensor([(int(L) + 127) // 128 for L in p.kv_lens]).view(-1, 1, 1, 1),
                       full, torch.full_like(full, -1)).contiguous()
    out3 = dv.sparse(block_idx=full.cuda(), topk=128).cpu().numpy()
    assert np.abs(out3 - dense_ref).max() <= TOL_BF16
    assert T.trtv_get_device_error() == 0
