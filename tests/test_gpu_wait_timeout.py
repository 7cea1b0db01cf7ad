"""The bounded waits' give-up path, made to happen on purpose: the test hook
trtv_test_withhold_pages stops every CTA's K producer after a few pages, so
the consumers' barrier waits run out (a short limit, a few milliseconds).  The
call must return promptly, the device error word must report
TRTV_DEVERR_TIMEOUT, and the next normal call in the same process must match
the oracle -- every kernel freed its tensor memory and left no copy in flight.

Source of the rule: "Eagle3 for M3 MSA path + CUDA graphs compatibility"
(fork PR #3), CUDA-graphs commit -- the path raises rather than waiting on
state that is not there; here a wait that cannot complete gives up, flags the
error and lets the kernel return.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_kv_gb300 as T
from speculative_decode_verify_kv_gb300 import workloads as W
from speculative_decode_verify_kv_gb300.runtime import DeviceVerify

pytestmark = pytest.mark.gpu

WAIT_US = 2000


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decode_verify_kv_gb300 import _build
    _build.build()
    T.load()
    T.trtv_get_device_error()  # clear
    yield
    T.trtv_test_withhold_pages(-1)


def starved(call, pages):
    """Run `call` with the K producers withholding after `pages` pages; return
    the error word and the wall time to completion."""
    T.trtv_get_device_error()
    torch.cuda.synchronize()
    T.trtv_test_withhold_pages(pages, WAIT_US)
    try:
        t0 = time.perf_counter()
        call()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        T.trtv_test_withhold_pages(-1)
    return T.trtv_get_device_error(), dt


def test_hook_rejects_bad_limits():
    with pytest.raises(T.TrtvError):
        T.trtv_test_withhold_pages(0, 0)
    with pytest.raises(T.TrtvError):
        T.trtv_test_withhold_pages(0, 3_000_000)
    T.trtv_test_withhold_pages(-1)


@pytest.mark.parametrize("Hq,Hk,dtype,pages", [
    (64, 4, W.BF16, 0),    # tcgen05 bf16 attention (64 rows): nothing arrives
    (64, 4, W.BF16, 2),    # ... after two pages, with work in every role
    (32, 4, W.BF16, 1),    # 32 rows
    (32, 4, W.FP8, 0),     # FP8 caches, 32 rows
    (64, 4, W.FP8, 3),     # FP8 caches, 64 rows
    (8, 8, W.BF16, 1),     # G = 1, mma.sync
])
def test_dense_wait_gives_up_and_next_call_is_exact(Hq, Hk, dtype, pages):
    p = W.make_problem(kv_lens=[3000, 700, 129, 4000, 33], qo_len=4, num_q_heads=Hq, num_kv_heads=Hk,
                       head_dim=128, kv_dtype=dtype, seed=90 + Hq + pages, slack_slots=3)
    dv = DeviceVerify(p, num_ctas=4, out_dtype="f32")   # dozens of pages per CTA
    err, dt = starved(dv.dense, pages)
    assert err & T.DEVERR_TIMEOUT
    assert dt < 1.0, f"starved call took {dt:.3f} s"
    out = dv.dense().cpu().numpy()
    ref, bad = oracle.verify_dense(oracle.Inputs(p))
    assert bad == 0
    assert np.abs(out - ref).max() <= (5e-2 if dtype == W.FP8 else 2e-2)
    assert T.trtv_get_device_error() == 0


@pytest.mark.parametrize("dtype", [W.BF16, W.FP8])
def test_proxy_and_select_give_up_and_recover(dtype):
    p = W.make_problem(kv_lens=[3000, 700, 129, 4000], qo_len=4, num_q_heads=64, num_kv_heads=4,
                       head_dim=128, kv_dtype=dtype, seed=95, topk=4, slack_slots=3, max_pages_per_req=40)
    dv = DeviceVerify(p, num_ctas=4)
    err, dt = starved(dv.proxy, 1)
    assert err & T.DEVERR_TIMEOUT and dt < 1.0
    err, dt = starved(dv.select_fused, 0)
    assert err & T.DEVERR_TIMEOUT and dt < 1.0
    sc = dv.proxy().cpu().numpy()
    ref, _ = oracle.proxy_score(oracle.Inputs(p))
    assert np.array_equal(np.isneginf(sc), np.isneginf(ref))
    f = np.isfinite(ref)
    assert np.abs(sc[f] - ref[f]).max() <= 1e-3
    idx = dv.select_fused().cpu().numpy()
    ref_i, _ = oracle.topk(oracle.Inputs(p), sc.astype(np.float64), p.topk)
    assert np.array_equal(idx, ref_i)
    assert T.trtv_get_device_error() == 0


def test_sparse_wait_gives_up_and_recovers():
    p = W.make_problem(kv_lens=[5000, 129, 4100], qo_len=8, num_q_heads=64, num_kv_heads=4,
                       head_dim=128, seed=97, topk=8, slack_slots=3, max_pages_per_req=40)
    dv = DeviceVerify(p, num_ctas=2, out_dtype="f32")
    dv.proxy()
    idx = dv.select().clone()
    err, dt = starved(dv.sparse, 1)
    assert err & T.DEVERR_TIMEOUT and dt < 1.0
    out = dv.sparse().cpu().numpy()
    ref, bad = oracle.sparse_attn(oracle.Inputs(p), idx.cpu().numpy())
    assert bad == 0 and np.abs(out - ref).max() <= 2e-2
    assert T.trtv_get_device_error() == 0
