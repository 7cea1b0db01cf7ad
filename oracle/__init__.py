"""fp64 CPU oracle for verify attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  The tests, the package's smoke check and the
benchmark's CPU-baseline leg use this module; the library's product path never
imports it.  The arithmetic lives in ``trtv_oracle.c`` (plain C, fp64); this
file only compiles it with gcc and marshals numpy arrays.

Inputs are the host tensors of :mod:`speculative_decode_verify_kv_gb300.workloads`
(bf16 passed as raw uint16 bits, FP8 as raw uint8 codes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "trtv_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_handle: Optional[ctypes.CDLL] = None

BF16, FP8 = 0, 1


class Problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("qo_len", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_pages_per_req", ctypes.c_int32),
                ("num_slots", ctypes.c_int32), ("slot_stride", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("sm_scale", ctypes.c_double),
                ("k_scale", ctypes.c_double), ("v_scale", ctypes.c_double)]


def _compile(src: str, out: str) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_lib/liboracle.so`` (OpenMP if gcc has it)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        return _compile(_SRC, _LIB)


def _bind(h: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.POINTER(Problem)
    vp = ctypes.c_void_p
    h.trtvo_bf16_to_double.restype = ctypes.c_double
    h.trtvo_bf16_to_double.argtypes = [ctypes.c_uint16]
    h.trtvo_e4m3_to_double.restype = ctypes.c_double
    h.trtvo_e4m3_to_double.argtypes = [ctypes.c_uint8]
    h.trtvo_element_offset.restype = ctypes.c_int64
    h.trtvo_element_offset.argtypes = [ctypes.c_int64] * 8
    h.trtvo_gather_head.argtypes = [P, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp]
    h.trtvo_subpage_view.argtypes = [P, vp, vp, vp, vp]
    h.trtvo_verify_dense.argtypes = [P, vp, vp, vp, vp, vp]
    h.trtvo_proxy_score.argtypes = [P, vp, vp, vp, vp, vp]
    h.trtvo_topk.argtypes = [P, vp, vp, ctypes.c_int, vp]
    h.trtvo_sparse_attn.argtypes = [P, vp, vp, vp, vp, vp, ctypes.c_int, vp]
    h.trtvo_e4m3_from_float.restype = ctypes.c_uint8
    h.trtvo_e4m3_from_float.argtypes = [ctypes.c_float]
    h.trtvo_stage_kv.argtypes = [P, vp, vp, vp, vp, vp]
    h.trtvo_flatten_page_table.argtypes = [P, vp, vp, vp, vp]
    h.trtvo_page_table_from_flat.argtypes = [P, vp, vp, vp]
    h.trtvo_draft_attn.argtypes = [P, vp, vp, vp, vp, vp, vp]
    h.trtvo_num_threads.restype = ctypes.c_int
    return h


def lib() -> ctypes.CDLL:
    global _handle
    if _handle is None:
        _handle = _bind(ctypes.CDLL(build()))
    return _handle


def load_variant(c_source: str, tag: str) -> "Oracle":
    """Compile ``c_source`` (a modified copy of the oracle, for tests that plant
    a mistake and check that the pins catch it) and return an Oracle on it."""
    import tempfile
    d = tempfile.mkdtemp(prefix=f"oracle_{tag}_")
    srcp = os.path.join(d, "oracle.c")
    with open(srcp, "w") as f:
        f.write(c_source)
    so = _compile(srcp, os.path.join(d, "liboracle.so"))
    return Oracle(_bind(ctypes.CDLL(so)))


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _np(t, dtype) -> np.ndarray:
    """torch tensor / numpy array -> contiguous numpy array viewed as ``dtype``."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype in (torch.bfloat16, torch.float16):
                t = t.view(torch.int16)
            elif t.dtype == torch.float8_e4m3fn:
                t = t.view(torch.uint8)
            t = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(t).view(dtype)


def problem_of(p, **over) -> Problem:
    """ctypes Problem from a workloads.VerifyProblem (fields overridable)."""
    f = dict(batch=p.batch, qo_len=p.qo_len, num_q_heads=p.num_q_heads,
             num_kv_heads=p.num_kv_heads, head_dim=p.head_dim,
             max_pages_per_req=p.max_pages_per_req, num_slots=p.num_slots,
             slot_stride=p.slot_stride, kv_dtype=FP8 if p.kv_dtype == "fp8_e4m3" else BF16,
             sm_scale=p.sm_scale, k_scale=p.k_scale, v_scale=p.v_scale)
    f.update(over)
    return Problem(**f)


class Inputs:
    """numpy views of a problem's tensors, kept alive for the C calls."""

    def __init__(self, p, *, q=None, pool=None, page_table=None, kv_lens=None, **over):
        self.P = problem_of(p, **over)
        self.q = _np(p.q if q is None else q, np.uint16)
        self.pool = _np(p.pool if pool is None else pool,
                        np.uint8 if self.P.kv_dtype == FP8 else np.uint16)
        self.pt = _np(p.page_table if page_table is None else page_table, np.int32)
        self.lens = _np(p.kv_lens if kv_lens is None else kv_lens, np.int32)


class Oracle:
    """The oracle's functions bound to one compiled library."""

    def __init__(self, handle: ctypes.CDLL):
        self.h = handle

    def bf16_to_double(self, bits: int) -> float:
        return self.h.trtvo_bf16_to_double(bits)

    def e4m3_to_double(self, code: int) -> float:
        return self.h.trtvo_e4m3_to_double(code)

    def element_offset(self, slot, stride, kv_heads, head_dim, p, h, kv, d) -> int:
        return self.h.trtvo_element_offset(slot, stride, kv_heads, head_dim, p, h, kv, d)

    def gather_head(self, x: Inputs, b: int, h: int):
        L = int(x.lens[b])
        D = x.P.head_dim
        K = np.zeros((max(L, 0), D), np.float64)
        V = np.zeros((max(L, 0), D), np.float64)
        rc = self.h.trtvo_gather_head(ctypes.byref(x.P), _ptr(x.pool), _ptr(x.pt), _ptr(x.lens),
                                     b, h, _ptr(K), _ptr(V))
        if rc != 0:
            raise ValueError("invalid request")
        return K, V

    def subpage_view(self, x: Inputs):
        n = 4 * x.P.max_pages_per_req
        k = np.zeros((x.P.batch, n), np.int32)
        v = np.zeros((x.P.batch, n), np.int32)
        bad = self.h.trtvo_subpage_view(ctypes.byref(x.P), _ptr(x.pt), _ptr(x.lens), _ptr(k), _ptr(v))
        return k, v, bad

    def verify_dense(self, x: Inputs):
        P = x.P
        out = np.zeros((P.batch * P.qo_len, P.num_q_heads, P.head_dim), np.float64)
        bad = self.h.trtvo_verify_dense(ctypes.byref(P), _ptr(x.q), _ptr(x.pool), _ptr(x.pt),
                                       _ptr(x.lens), _ptr(out))
        return out, bad

    def proxy_score(self, x: Inputs):
        P = x.P
        s = np.zeros((P.batch, P.qo_len, P.num_kv_heads, P.max_pages_per_req), np.float64)
        bad = self.h.trtvo_proxy_score(ctypes.byref(P), _ptr(x.q), _ptr(x.pool), _ptr(x.pt),
                                      _ptr(x.lens), _ptr(s))
        return s, bad

    def topk(self, x: Inputs, scores: np.ndarray, k: int):
        P = x.P
        s = np.ascontiguousarray(scores, dtype=np.float64)
        idx = np.zeros((P.batch, P.qo_len, P.num_kv_heads, k), np.int32)
        bad = self.h.trtvo_topk(ctypes.byref(P), _ptr(x.lens), _ptr(s), k, _ptr(idx))
        return idx, bad

    def sparse_attn(self, x: Inputs, idx: np.ndarray, k: Optional[int] = None):
        P = x.P
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        k = idx.shape[-1] if k is None else k
        out = np.zeros((P.batch * P.qo_len, P.num_q_heads, P.head_dim), np.float64)
        bad = self.h.trtvo_sparse_attn(ctypes.byref(P), _ptr(x.q), _ptr(x.pool), _ptr(x.pt),
                                      _ptr(x.lens), _ptr(idx), k, _ptr(out))
        return out, bad

    def e4m3_from_float(self, x: float) -> int:
        return int(self.h.trtvo_e4m3_from_float(x))

    def stage_kv(self, x: Inputs, k_new, v_new):
        """Stage the qo_len new tokens' K and V ([B*T, Hk, D] bf16) into a copy
        of the pool; returns (new pool, requests not staged)."""
        P = x.P
        kn = _np(k_new, np.uint16)
        vn = _np(v_new, np.uint16)
        pool = x.pool.copy()
        bad = self.h.trtvo_stage_kv(ctypes.byref(P), _ptr(kn), _ptr(vn), _ptr(x.pt), _ptr(x.lens),
                                    _ptr(pool))
        return pool, bad

    def flatten_page_table(self, x: Inputs, flat_init=None):
        """Flat table [B*max_pages] and indptr [B+1] restaged from the padded
        table and the lengths; entries past indptr[B] keep ``flat_init``
        (zeros by default).  Returns (flat, indptr, invalid requests)."""
        P = x.P
        n = P.batch * P.max_pages_per_req
        flat = (np.zeros(n, np.int32) if flat_init is None
                else np.array(_np(flat_init, np.int32), dtype=np.int32).reshape(-1).copy())
        indptr = np.zeros(P.batch + 1, np.int32)
        bad = self.h.trtvo_flatten_page_table(ctypes.byref(P), _ptr(x.pt), _ptr(x.lens), _ptr(flat),
                                              _ptr(indptr))
        return flat, indptr, bad

    def page_table_from_flat(self, x: Inputs, flat):
        """Padded table [B, max_pages] from a flat table whose row bases come
        from the lengths.  Returns (page_table, invalid requests)."""
        P = x.P
        f = _np(flat, np.int32)
        pt = np.zeros((P.batch, P.max_pages_per_req), np.int32)
        bad = self.h.trtvo_page_table_from_flat(ctypes.byref(P), _ptr(f), _ptr(x.lens), _ptr(pt))
        return pt, bad

    def draft_attn(self, x: Inputs, k_sub, v_sub):
        """Attention through the P32 sub-page tables k_sub / v_sub [B, 4*max_pages]."""
        P = x.P
        ks = _np(k_sub, np.int32)
        vs = _np(v_sub, np.int32)
        out = np.zeros((P.batch * P.qo_len, P.num_q_heads, P.head_dim), np.float64)
        bad = self.h.trtvo_draft_attn(ctypes.byref(P), _ptr(x.q), _ptr(x.pool), _ptr(ks), _ptr(vs),
                                      _ptr(x.lens), _ptr(out))
        return out, bad

    def num_threads(self) -> int:
        return self.h.trtvo_num_threads()


_default: Optional[Oracle] = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(lib())
    return _default


def __getattr__(name):
    # module-level access to the default oracle's functions: oracle.verify_dense(...)
    if name in Oracle.__dict__ and not name.startswith("_"):
        return getattr(default(), name)
    raise AttributeError(name)
