"""Python binding of the GB300 verify-attention library (``include/trtv.h``).

Argument marshalling only: each function takes torch CUDA tensors (or raw
device pointers), converts them to pointers and sizes, and calls the C entry
point of the same name in ``_lib/libtrtv.so``.  Every step of the path runs in
the library's CUDA kernels; there is no fallback.  Importing the package does
not need a GPU, but calling a compute function without the built library or
without a GPU raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

__all__ = [
    "TRTV_OK", "TRTV_BF16", "TRTV_FP8_E4M3", "TRTV_F32", "TrtvError", "Geom", "load",
    "trtv_subpage_view", "trtv_workspace_bytes", "trtv_verify_dense", "trtv_msa_proxy_score",
    "trtv_msa_topk", "trtv_msa_sparse_attn", "trtv_get_device_error", "trtv_version",
    "trtv_verify_dense_noalloc", "trtv_stage_kv", "trtv_flatten_page_table",
    "trtv_page_table_from_flat", "trtv_workspace_bytes_flat", "trtv_verify_dense_flat",
    "trtv_draft_attn_p32", "trtv_msa_select", "trtv_msa_verify", "trtv_status_string",
    "trtv_test_withhold_pages", "geom_of", "EXPORTS",
]

TRTV_OK, TRTV_ERR_INVALID_ARG, TRTV_ERR_UNSUPPORTED, TRTV_ERR_CUDA, TRTV_ERR_WORKSPACE = range(5)
TRTV_BF16, TRTV_FP8_E4M3, TRTV_F32 = 0, 1, 2
DEVERR_KV_LEN, DEVERR_PAGE_ID, DEVERR_BLOCK_IDX, DEVERR_TIMEOUT = 1, 2, 4, 8

# every function the C header declares
EXPORTS = ("trtv_status_string", "trtv_version", "trtv_subpage_view", "trtv_workspace_bytes",
           "trtv_verify_dense", "trtv_verify_dense_noalloc", "trtv_msa_proxy_score", "trtv_msa_topk",
           "trtv_msa_sparse_attn", "trtv_stage_kv", "trtv_flatten_page_table",
           "trtv_page_table_from_flat", "trtv_workspace_bytes_flat", "trtv_verify_dense_flat",
           "trtv_draft_attn_p32", "trtv_msa_select", "trtv_msa_verify", "trtv_test_withhold_pages",
           "trtv_get_device_error")


class TrtvError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


class Geom(ctypes.Structure):
    """Mirror of ``trtv_geom``."""
    _fields_ = [("batch", ctypes.c_int32), ("qo_len", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_pages_per_req", ctypes.c_int32),
                ("num_slots", ctypes.c_int32), ("slot_stride", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("sm_scale", ctypes.c_float),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
                ("num_ctas", ctypes.c_int32)]


_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load ``libtrtv.so`` (building it first when asked).  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError(f"libtrtv.so is not built ({path}); run __graft_entry__.build() "
                              "or python -m speculative_decode_verify_kv_gb300._build")
        _build.build()
    h = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    G = ctypes.POINTER(Geom)
    h.trtv_status_string.restype = ctypes.c_char_p
    h.trtv_status_string.argtypes = [ctypes.c_int]
    h.trtv_version.restype = i32
    h.trtv_version.argtypes = []
    h.trtv_subpage_view.restype = ctypes.c_int
    h.trtv_subpage_view.argtypes = [G, vp, vp, vp, vp, vp]
    h.trtv_workspace_bytes.restype = sz
    h.trtv_workspace_bytes.argtypes = [G, i32]
    h.trtv_verify_dense.restype = ctypes.c_int
    h.trtv_verify_dense.argtypes = [G, vp, vp, vp, vp, vp, i32, vp, sz, vp]
    h.trtv_verify_dense_noalloc.restype = ctypes.c_int
    h.trtv_verify_dense_noalloc.argtypes = [G, vp, vp, vp, vp, vp, i32, vp]
    h.trtv_msa_proxy_score.restype = ctypes.c_int
    h.trtv_msa_proxy_score.argtypes = [G, vp, vp, vp, vp, vp, vp]
    h.trtv_msa_topk.restype = ctypes.c_int
    h.trtv_msa_topk.argtypes = [G, vp, vp, i32, vp, vp]
    h.trtv_msa_sparse_attn.restype = ctypes.c_int
    h.trtv_msa_sparse_attn.argtypes = [G, vp, vp, vp, vp, vp, i32, vp, i32, vp, sz, vp]
    h.trtv_stage_kv.restype = ctypes.c_int
    h.trtv_stage_kv.argtypes = [G, vp, vp, vp, vp, vp, vp]
    h.trtv_flatten_page_table.restype = ctypes.c_int
    h.trtv_flatten_page_table.argtypes = [G, vp, vp, vp, vp, vp]
    h.trtv_page_table_from_flat.restype = ctypes.c_int
    h.trtv_page_table_from_flat.argtypes = [G, vp, vp, vp, vp]
    h.trtv_workspace_bytes_flat.restype = sz
    h.trtv_workspace_bytes_flat.argtypes = [G]
    h.trtv_verify_dense_flat.restype = ctypes.c_int
    h.trtv_verify_dense_flat.argtypes = [G, vp, vp, vp, vp, vp, i32, vp, sz, vp]
    h.trtv_draft_attn_p32.restype = ctypes.c_int
    h.trtv_draft_attn_p32.argtypes = [G, vp, vp, vp, vp, vp, vp, i32, vp, sz, vp]
    h.trtv_msa_select.restype = ctypes.c_int
    h.trtv_msa_select.argtypes = [G, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    h.trtv_msa_verify.restype = ctypes.c_int
    h.trtv_msa_verify.argtypes = [G, vp, vp, vp, vp, i32, vp, vp, vp, i32, vp, sz, vp]
    h.trtv_get_device_error.restype = ctypes.c_int
    h.trtv_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
    h.trtv_test_withhold_pages.restype = ctypes.c_int
    h.trtv_test_withhold_pages.argtypes = [i32, ctypes.c_uint32]
    _lib = h
    return h


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int) -> None:
    if st != TRTV_OK:
        raise TrtvError(fn, st, load().trtv_status_string(st).decode())


def geom_of(p, num_ctas: int = 0, **over) -> Geom:
    """Geom from a workloads.VerifyProblem-like object (fields overridable)."""
    f = dict(batch=p.batch, qo_len=p.qo_len, num_q_heads=p.num_q_heads,
             num_kv_heads=p.num_kv_heads, head_dim=p.head_dim,
             max_pages_per_req=p.max_pages_per_req, num_slots=p.num_slots,
             slot_stride=p.slot_stride,
             kv_dtype=TRTV_FP8_E4M3 if p.kv_dtype == "fp8_e4m3" else TRTV_BF16,
             sm_scale=p.sm_scale, k_scale=p.k_scale, v_scale=p.v_scale, num_ctas=num_ctas)
    f.update(over)
    return Geom(**f)


def trtv_version() -> int:
    return load().trtv_version()


def trtv_status_string(st: int) -> str:
    return load().trtv_status_string(st).decode()


def trtv_workspace_bytes(geom: Geom, topk: int = 0) -> int:
    return load().trtv_workspace_bytes(ctypes.byref(geom), topk)


def trtv_subpage_view(geom: Geom, page_table, kv_lens, k_sub, v_sub, stream=None) -> None:
    _check("trtv_subpage_view", load().trtv_subpage_view(
        ctypes.byref(geom), _ptr(page_table), _ptr(kv_lens), _ptr(k_sub), _ptr(v_sub),
        _stream(stream)))


def trtv_verify_dense(geom: Geom, q, kv_pool, page_table, kv_lens, out, out_dtype: int,
                      workspace, ws_bytes: int, stream=None) -> None:
    _check("trtv_verify_dense", load().trtv_verify_dense(
        ctypes.byref(geom), _ptr(q), _ptr(kv_pool), _ptr(page_table), _ptr(kv_lens), _ptr(out),
        out_dtype, _ptr(workspace), ws_bytes, _stream(stream)))


def trtv_verify_dense_noalloc(geom: Geom, q, kv_pool, page_table, kv_lens, out, out_dtype: int,
                              stream=None) -> None:
    """trtv_verify_dense with the library's static device scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    _check("trtv_verify_dense_noalloc", load().trtv_verify_dense_noalloc(
        ctypes.byref(geom), _ptr(q), _ptr(kv_pool), _ptr(page_table), _ptr(kv_lens), _ptr(out),
        out_dtype, _stream(stream)))


def trtv_msa_proxy_score(geom: Geom, q, kv_pool, page_table, kv_lens, scores, stream=None) -> None:
    _check("trtv_msa_proxy_score", load().trtv_msa_proxy_score(
        ctypes.byref(geom), _ptr(q), _ptr(kv_pool), _ptr(page_table), _ptr(kv_lens),
        _ptr(scores), _stream(stream)))


def trtv_msa_topk(geom: Geom, scores, kv_lens, topk: int, block_idx, stream=None) -> None:
    _check("trtv_msa_topk", load().trtv_msa_topk(
        ctypes.byref(geom), _ptr(scores), _ptr(kv_lens), topk, _ptr(block_idx), _stream(stream)))


def trtv_msa_select(geom: Geom, q, kv_pool, page_table, kv_lens, topk: int, scores, block_idx,
                    workspace, ws_bytes: int, stream=None) -> None:
    """Proxy scores and per-token top-k in one call (fused where the tcgen05
    proxy kernel applies)."""
    _check("trtv_msa_select", load().trtv_msa_select(
        ctypes.byref(geom), _ptr(q), _ptr(kv_pool), _ptr(page_table), _ptr(kv_lens), topk,
        _ptr(scores), _ptr(block_idx), _ptr(workspace), ws_bytes, _stream(stream)))


def trtv_msa_verify(geom: Geom, q, kv_pool, page_table, kv_lens, topk: int, scores, block_idx, out,
                    out_dtype: int, workspace, ws_bytes: int, stream=None) -> None:
    """Proxy scores, per-token top-k and sparse attention in one call (the
    fused select builds the sparse plan where it applies)."""
    _check("trtv_msa_verify", load().trtv_msa_verify(
        ctypes.byref(geom), _ptr(q), _ptr(kv_pool), _ptr(page_table), _ptr(kv_lens), topk,
        _ptr(scores), _ptr(block_idx), _ptr(out), out_dtype, _ptr(workspace), ws_bytes, _stream(stream)))


def trtv_msa_sparse_attn(geom: Geom, q, kv_pool, page_table, kv_lens, block_idx, topk: int, out,
                         out_dtype: int, workspace, ws_bytes: int, stream=None) -> None:
    _check("trtv_msa_sparse_attn", load().trtv_msa_sparse_attn(
        ctypes.byref(geom), _ptr(q), _ptr(kv_pool), _ptr(page_table), _ptr(kv_lens),
        _ptr(block_idx), topk, _ptr(out), out_dtype, _ptr(workspace), ws_bytes, _stream(stream)))


def trtv_stage_kv(geom: Geom, k_new, v_new, kv_pool, page_table, kv_lens, stream=None) -> None:
    _check("trtv_stage_kv", load().trtv_stage_kv(
        ctypes.byref(geom), _ptr(k_new), _ptr(v_new), _ptr(kv_pool), _ptr(page_table), _ptr(kv_lens),
        _stream(stream)))


def trtv_flatten_page_table(geom: Geom, page_table, kv_lens, flat, indptr=None, stream=None) -> None:
    """Restage the flat (CSR) page table from the padded one and the lengths."""
    _check("trtv_flatten_page_table", load().trtv_flatten_page_table(
        ctypes.byref(geom), _ptr(page_table), _ptr(kv_lens), _ptr(flat), _ptr(indptr),
        _stream(stream)))


def trtv_page_table_from_flat(geom: Geom, flat, kv_lens, page_table, stream=None) -> None:
    """Padded page table from a flat one whose row bases follow the lengths."""
    _check("trtv_page_table_from_flat", load().trtv_page_table_from_flat(
        ctypes.byref(geom), _ptr(flat), _ptr(kv_lens), _ptr(page_table), _stream(stream)))


def trtv_workspace_bytes_flat(geom: Geom) -> int:
    return load().trtv_workspace_bytes_flat(ctypes.byref(geom))


def trtv_verify_dense_flat(geom: Geom, q, kv_pool, flat, kv_lens, out, out_dtype: int, workspace,
                           ws_bytes: int, stream=None) -> None:
    _check("trtv_verify_dense_flat", load().trtv_verify_dense_flat(
        ctypes.byref(geom), _ptr(q), _ptr(kv_pool), _ptr(flat), _ptr(kv_lens), _ptr(out), out_dtype,
        _ptr(workspace), ws_bytes, _stream(stream)))


def trtv_draft_attn_p32(geom: Geom, q, kv_pool, k_sub, v_sub, kv_lens, out, out_dtype: int,
                        workspace, ws_bytes: int, stream=None) -> None:
    """Attention read through the P32 sub-page tables (the drafter's view)."""
    _check("trtv_draft_attn_p32", load().trtv_draft_attn_p32(
        ctypes.byref(geom), _ptr(q), _ptr(kv_pool), _ptr(k_sub), _ptr(v_sub), _ptr(kv_lens),
        _ptr(out), out_dtype, _ptr(workspace), ws_bytes, _stream(stream)))


def trtv_test_withhold_pages(pages: int, wait_us: int = 0) -> None:
    """Test hook of the bounded waits: K producers stop after ``pages`` pages
    and every wait gives up after ``wait_us``; ``pages < 0`` restores normal
    operation."""
    _check("trtv_test_withhold_pages", load().trtv_test_withhold_pages(pages, wait_us))


def trtv_get_device_error(stream=None) -> int:
    v = ctypes.c_int32(0)
    _check("trtv_get_device_error", load().trtv_get_device_error(ctypes.byref(v), _stream(stream)))
    return v.value
