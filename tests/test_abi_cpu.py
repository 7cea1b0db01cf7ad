"""The C-ABI library on the CPU: it loads, exports every function the header
declares, and its host-side validation rejects bad arguments before any CUDA
call (no GPU needed; num_ctas > 0 keeps the planner off the device)."""
import ctypes
import os
import re

import pytest

import speculative_decode_verify_kv_gb300 as T
from speculative_decode_verify_kv_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "trtv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return T.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(trtv_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("trtv_verify_dense", "trtv_msa_proxy_score", "trtv_msa_topk", "trtv_msa_sparse_attn",
              "trtv_subpage_view"):
        assert n in names
    assert set(names) == set(T.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert T.trtv_version() >= 100
    assert T.trtv_status_string(0) == "ok"
    assert "workspace" in T.trtv_status_string(4)


def geom(**over):
    g = dict(batch=2, qo_len=4, num_q_heads=8, num_kv_heads=2, head_dim=64, max_pages_per_req=3,
             num_slots=8, slot_stride=2, kv_dtype=0, sm_scale=0.125, k_scale=1.0, v_scale=1.0,
             num_ctas=4)
    g.update(over)
    return T.Geom(**g)


@pytest.mark.parametrize("over,status", [
    (dict(batch=0), 1), (dict(qo_len=0), 1), (dict(num_q_heads=6, num_kv_heads=4), 1),
    (dict(slot_stride=1), 1), (dict(max_pages_per_req=0), 1), (dict(kv_dtype=7), 1),
    (dict(sm_scale=0.0), 1), (dict(k_scale=-1.0), 1), (dict(v_scale=float("inf")), 1),
    (dict(num_ctas=-1), 1), (dict(head_dim=96), 2), (dict(kv_dtype=1, head_dim=64), 2),
    (dict(qo_len=33), 2), (dict(num_q_heads=64, num_kv_heads=1, qo_len=4), 2),
    (dict(num_slots=1 << 20, num_kv_heads=2, slot_stride=8), 2),
])
def test_geometry_validation(lib, over, status):
    g = geom(**over)
    assert lib.trtv_workspace_bytes(ctypes.byref(g), 0) == 0
    st = lib.trtv_verify_dense(ctypes.byref(g), 16, 16, 16, 16, 16, 0, 256, 1 << 30, None)
    assert st == status


def test_workspace_size_and_checks(lib):
    g = geom()
    need = lib.trtv_workspace_bytes(ctypes.byref(g), 0)
    # 2 partial slots per CTA x 16 padded rows x (64 outputs + 1 lse) floats + one 32-byte
    # split descriptor per CTA, each region 256-byte aligned
    assert need == 2 * 4 * 16 * 64 * 4 + 512 + 256
    need_sparse = lib.trtv_workspace_bytes(ctypes.byref(g), 2)
    assert need_sparse > need
    # too small / misaligned workspace is rejected on the host
    assert lib.trtv_verify_dense(ctypes.byref(g), 16, 16, 16, 16, 16, 0, 256, need - 1, None) == 4
    assert lib.trtv_verify_dense(ctypes.byref(g), 16, 16, 16, 16, 16, 0, 128, need, None) == 4
    # null or misaligned pointers
    assert lib.trtv_verify_dense(ctypes.byref(g), 0, 16, 16, 16, 16, 0, 256, need, None) == 1
    assert lib.trtv_verify_dense(ctypes.byref(g), 16, 8, 16, 16, 16, 0, 256, need, None) == 1
    assert lib.trtv_verify_dense(ctypes.byref(g), 16, 16, 16, 16, 16, 5, 256, need, None) == 1
    assert lib.trtv_msa_sparse_attn(ctypes.byref(g), 16, 16, 16, 16, 0, 2, 16, 0, 256, need_sparse, None) == 1
    assert lib.trtv_msa_sparse_attn(ctypes.byref(g), 16, 16, 16, 16, 16, 0, 16, 0, 256, need_sparse, None) == 1
    assert lib.trtv_msa_topk(ctypes.byref(g), 16, 16, 0, 16, None) == 1
    assert lib.trtv_msa_topk(ctypes.byref(g), 16, 16, 2000, 16, None) == 1
    assert lib.trtv_subpage_view(ctypes.byref(g), 0, 16, 16, 16, None) == 1
    big = geom(num_q_heads=64, num_kv_heads=2)  # group 32 > 16: no proxy
    assert lib.trtv_msa_proxy_score(ctypes.byref(big), 16, 16, 16, 16, 16, None) == 2
    assert lib.trtv_get_device_error(None, None) == 1


def test_stage_kv_argument_checks(lib):
    g = geom()
    # null or misaligned pointers are rejected on the host, before any launch
    assert lib.trtv_stage_kv(ctypes.byref(g), 0, 16, 16, 16, 16, None) == 1
    assert lib.trtv_stage_kv(ctypes.byref(g), 16, 16, 0, 16, 16, None) == 1
    assert lib.trtv_stage_kv(ctypes.byref(g), 8, 16, 16, 16, 16, None) == 1
    assert lib.trtv_stage_kv(ctypes.byref(g), 16, 16, 24, 16, 16, None) == 1
    bad = geom(slot_stride=1)
    assert lib.trtv_stage_kv(ctypes.byref(bad), 16, 16, 16, 16, 16, None) == 1


def test_flat_table_and_draft_argument_checks(lib):
    g = geom()
    need = lib.trtv_workspace_bytes(ctypes.byref(g), 0)
    # the rebuilt padded table (2 x 3 int32) takes one more 256-byte region
    need_flat = lib.trtv_workspace_bytes_flat(ctypes.byref(g))
    assert need_flat == need + 256
    assert lib.trtv_verify_dense_flat(ctypes.byref(g), 16, 16, 16, 16, 16, 0, 256, need, None) == 4
    assert lib.trtv_verify_dense_flat(ctypes.byref(g), 16, 16, 0, 16, 16, 0, 256, need_flat, None) == 1
    assert lib.trtv_verify_dense_flat(ctypes.byref(g), 16, 16, 16, 0, 16, 0, 256, need_flat, None) == 1
    assert lib.trtv_draft_attn_p32(ctypes.byref(g), 16, 16, 0, 16, 16, 16, 0, 256, need, None) == 1
    assert lib.trtv_draft_attn_p32(ctypes.byref(g), 16, 16, 16, 0, 16, 16, 0, 256, need, None) == 1
    assert lib.trtv_draft_attn_p32(ctypes.byref(g), 16, 16, 16, 16, 16, 16, 0, 256, need - 1, None) == 4
    assert lib.trtv_draft_attn_p32(ctypes.byref(g), 16, 8, 16, 16, 16, 16, 0, 256, need, None) == 1
    assert lib.trtv_flatten_page_table(ctypes.byref(g), 0, 16, 16, 16, None) == 1
    assert lib.trtv_flatten_page_table(ctypes.byref(g), 16, 16, 0, None, None) == 1
    assert lib.trtv_page_table_from_flat(ctypes.byref(g), 16, 16, 0, None) == 1
    assert lib.trtv_page_table_from_flat(ctypes.byref(geom(batch=0)), 16, 16, 16, None) == 1
    assert lib.trtv_flatten_page_table(ctypes.byref(geom(batch=70000)), 16, 16, 16, None, None) == 2
    assert lib.trtv_workspace_bytes_flat(ctypes.byref(geom(batch=0))) == 0


def test_msa_select_argument_checks(lib):
    g = geom()
    need = lib.trtv_workspace_bytes(ctypes.byref(g), 2)
    # null outputs / bad k / small workspace are rejected on the host
    assert lib.trtv_msa_select(ctypes.byref(g), 16, 16, 16, 16, 2, 16, 0, 256, need, None) == 1
    assert lib.trtv_msa_select(ctypes.byref(g), 16, 16, 16, 16, 0, 16, 16, 256, need, None) == 1
    assert lib.trtv_msa_select(ctypes.byref(g), 16, 16, 16, 16, 2000, 16, 16, 256, need, None) == 1
    assert lib.trtv_msa_select(ctypes.byref(g), 16, 16, 16, 16, 2, 16, 16, 256, need - 1, None) == 4
    assert lib.trtv_msa_select(ctypes.byref(g), 16, 16, 16, 16, 2, 16, 16, 128, need, None) == 4
    assert lib.trtv_msa_select(ctypes.byref(g), 16, 16, 16, 16, 2, 0, 16, 256, need, None) == 1
    big = geom(num_q_heads=64, num_kv_heads=2)  # group 32 > 16: no proxy
    assert lib.trtv_msa_select(ctypes.byref(big), 16, 16, 16, 16, 2, 16, 16, 256, 1 << 30, None) == 2


def test_header_is_plain_c(lib, tmp_path):
    """The boundary is a C ABI: the header compiles as strict C99 on its own,
    and a C program links every declared entry point against the library."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use.c"
    calls = "\n".join(f"  p[{i}] = (void (*)(void)){n};" for i, n in enumerate(declared_functions()))
    src.write_text('#include "trtv.h"\n'
                   f"int main(void) {{\n  void (*p[{len(declared_functions())}])(void);\n{calls}\n"
                   "  return p[0] == 0;\n}\n")
    inc = os.path.join(os.path.dirname(HEADER))
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I" + inc,
                        str(src), "-o", str(tmp_path / "use"), _build.LIB, "-Wl,-rpath," + os.path.dirname(_build.LIB)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
