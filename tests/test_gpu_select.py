"""Proxy scores + per-token top-k in one call (trtv_msa_select) against the
two-call path and the oracle: scores identical to trtv_msa_proxy_score's,
indices bit-exact (the oracle's selection run on the GPU's fp32 scores).  The
whole MSA step in one call (trtv_msa_verify, whose fused select also builds
the sparse plan) against select + sparse attention: bit-identical."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_kv_gb300 as T
from speculative_decode_verify_kv_gb300 import workloads as W
from speculative_decode_verify_kv_gb300.runtime import DeviceVerify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decode_verify_kv_gb300 import _build
    _build.build()
    T.load()
    T.trtv_get_device_error()  # clear


def _two_call(dv):
    dv.proxy()
    dv.select()
    torch.cuda.synchronize()
    return dv.scores.clone(), dv.block_idx.clone()


def _fused(dv):
    dv.scores.fill_(float("nan"))
    dv.block_idx.fill_(-7)
    dv.select_fused()
    torch.cuda.synchronize()
    return dv.scores.clone(), dv.block_idx.clone()


@pytest.mark.parametrize("Hq,Hk,Tq,dtype,num_ctas", [
    (64, 4, 4, W.BF16, 0),     # tcgen05 proxy, top-k fused (64 rows)
    (64, 4, 4, W.BF16, 1),     # one CTA completes every sequence
    (32, 4, 4, W.BF16, 7),     # sequences cut across CTAs
    (16, 2, 8, W.BF16, 150),   # many CTAs per sequence
    (32, 4, 4, W.FP8, 5),      # FP8: proxy kernel, then the top-k kernel
])
def test_select_equals_two_calls(Hq, Hk, Tq, dtype, num_ctas):
    p = W.make_problem(kv_lens=[3000, 129, 2, 5000, 700, 40], qo_len=Tq, num_q_heads=Hq, num_kv_heads=Hk,
                       head_dim=128, kv_dtype=dtype, seed=Hq + Tq + num_ctas, topk=8, max_pages_per_req=48)
    dv = DeviceVerify(p, num_ctas=num_ctas)
    s2, i2 = _two_call(dv)
    T.trtv_get_device_error()
    s1, i1 = _fused(dv)
    assert T.trtv_get_device_error() & T.DEVERR_KV_LEN          # request 2: kv_len < qo_len
    assert torch.equal(s1, s2)
    assert torch.equal(i1, i2)
    ref, _ = oracle.topk(oracle.Inputs(p), s1.cpu().double().numpy(), p.topk)
    assert np.array_equal(i1.cpu().numpy(), ref)
    assert torch.all(i1[2] == -1)


def test_select_long_rows_and_ties():
    """Rows past the register-key capacity (1100 blocks) and equal scores
    (a K page shared by many blocks): fused = two calls = oracle."""
    p = W.make_problem(kv_lens=[1100 * 128, 900 * 128 + 5], qo_len=4, num_q_heads=16, num_kv_heads=1,
                       head_dim=128, seed=71, topk=40, max_pages_per_req=1100)
    pt = p.page_table.clone()
    pt[1, 100:400] = pt[1, 99]       # identical pages -> tied scores
    p = p.with_(page_table=pt)
    dv = DeviceVerify(p, num_ctas=0)
    s2, i2 = _two_call(dv)
    s1, i1 = _fused(dv)
    assert torch.equal(s1, s2) and torch.equal(i1, i2)
    ref, _ = oracle.topk(oracle.Inputs(p), s1.cpu().double().numpy(), p.topk)
    assert np.array_equal(i1.cpu().numpy(), ref)
    assert T.trtv_get_device_error() == 0


def test_select_then_sparse_under_graph_replay():
    """Capture select + sparse once; replays with mutated lengths match the
    oracle's sparse attention on the replay's own indices."""
    p = W.make_problem(kv_lens=[2000, 900, 4000], qo_len=4, num_q_heads=64, num_kv_heads=4, head_dim=128,
                       seed=72, topk=6, max_pages_per_req=40, out_dtype="f32")
    dv = DeviceVerify(p, out_dtype="f32")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dv.msa_fused(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dv.msa_fused()
    for lens in ([2000, 900, 4000], [5120, 128, 129], [3, 4096, 700]):
        lens_t = torch.tensor(lens, dtype=torch.int32)
        dv.kv_lens.copy_(lens_t)
        graph.replay()
        torch.cuda.synchronize()
        x = oracle.Inputs(p, kv_lens=lens_t)
        idx = dv.block_idx.cpu().numpy()
        ref_idx, _ = oracle.topk(x, dv.scores.cpu().double().numpy(), p.topk)
        assert np.array_equal(idx, ref_idx)
        ref, _ = oracle.sparse_attn(x, idx)
        assert np.abs(dv.out.cpu().numpy() - ref).max() <= 2e-2
        T.trtv_get_device_error()


@pytest.mark.parametrize("Hq,Hk,Tq,dtype,num_ctas,max_pages", [
    (64, 4, 4, W.BF16, 0, 48),      # fused select builds the plan (64 rows)
    (64, 4, 4, W.BF16, 1, 48),      # one CTA selects and plans every sequence
    (32, 4, 4, W.BF16, 7, 48),      # 32 rows: position-major attention
    (16, 2, 8, W.BF16, 150, 48),    # many CTAs per sequence
    (64, 4, 8, W.BF16, 5, 48),      # 128 rows
    (64, 4, 4, W.BF16, 0, 2040),    # too many pages per request: plan kernel
    (32, 4, 4, W.FP8, 5, 48),       # FP8: proxy + top-k kernels + plan kernel
])
def test_msa_verify_equals_select_then_sparse(Hq, Hk, Tq, dtype, num_ctas, max_pages):
    p = W.make_problem(kv_lens=[3000, 129, 2, 5000, 700, 40], qo_len=Tq, num_q_heads=Hq, num_kv_heads=Hk,
                       head_dim=128, kv_dtype=dtype, seed=Hq + Tq + num_ctas + 5, topk=8,
                       max_pages_per_req=max_pages, out_dtype="f32")
    dv = DeviceVerify(p, num_ctas=num_ctas, out_dtype="f32")
    dv.select_fused()
    dv.sparse()
    torch.cuda.synchronize()
    i2, o2 = dv.block_idx.clone(), dv.out.clone()
    T.trtv_get_device_error()
    dv.block_idx.fill_(-7)
    dv.out.fill_(float("nan"))
    dv.workspace.fill_(0xAB)  # the one-call path needs no workspace contents
    dv.msa_verify()
    torch.cuda.synchronize()
    assert T.trtv_get_device_error() & T.DEVERR_KV_LEN          # request 2: kv_len < qo_len
    assert torch.equal(dv.block_idx, i2)
    assert torch.equal(dv.out, o2)
    ref, _ = oracle.sparse_attn(oracle.Inputs(p), i2.cpu().numpy())
    assert np.abs(dv.out.cpu().numpy() - ref).max() <= 2e-2
