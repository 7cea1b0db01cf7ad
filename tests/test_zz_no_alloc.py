"""trtv_verify_dense_noalloc: the dense verify entry point for callers that
cannot allocate device memory (its scratch is a static device array inside the
library).  Its output must match trtv_verify_dense with a caller workspace on
calls in a row, and the calls must leave the device's free memory unchanged.
This file is collected last, so a run that stops at the first failure has
already run every other test."""
import pytest
import torch

import speculative_decode_verify_kv_gb300 as T
from speculative_decode_verify_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 2e-2  # max-abs tolerance of the dense parity tests (bf16 K/V)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decode_verify_kv_gb300 import _build
    _build.build()
    T.load()


@pytest.mark.parametrize("lens,Hq,Hk,D", [
    ([1000, 37, 513, 4, 2000], 32, 4, 128),
    ([3000, 129, 77], 8, 2, 64),
])
def test_noalloc_matches_workspace_entry_point(lens, Hq, Hk, D):
    from speculative_decode_verify_kv_gb300.runtime import DeviceVerify
    p = W.make_problem(kv_lens=lens, qo_len=4, num_q_heads=Hq, num_kv_heads=Hk, head_dim=D,
                       seed=len(lens) + D, slack_slots=5)
    dv = DeviceVerify(p, out_dtype="f32")
    ref = dv.dense().clone()
    outs = [torch.full_like(dv.out, float("nan")) for _ in range(3)]
    torch.cuda.synchronize()
    free = []
    for out in outs:  # nothing but the calls between the readings of free memory
        T.trtv_verify_dense_noalloc(dv.geom, dv.q, dv.pool, dv.page_table, dv.kv_lens, out, T.TRTV_F32)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    # the entry point allocates nothing: device memory stays as it was after the first call
    assert free[1] == free[0] and free[2] == free[0], free
    for out in outs:
        assert torch.isfinite(out).all()
        assert (out - ref).abs().max().item() <= TOL
    assert T.trtv_get_device_error() == 0


def test_noalloc_rejects_geometry_beyond_its_scratch():
    g = T.Geom(batch=8, qo_len=8, num_q_heads=128, num_kv_heads=8, head_dim=128, max_pages_per_req=4,
               num_slots=64, slot_stride=2, kv_dtype=0, sm_scale=0.1, k_scale=1.0, v_scale=1.0,
               num_ctas=1024)
    assert T.trtv_workspace_bytes(g, 0) > 24 << 20
    dummy = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(T.TrtvError) as e:
        T.trtv_verify_dense_noalloc(g, dummy, dummy, dummy, dummy, dummy, T.TRTV_F32)
    assert e.value.status == T.TRTV_ERR_WORKSPACE
