"""Prepare-time buffers for verify calls on one GPU.

Everything a verify step touches is allocated once here (inputs copied to the
device, outputs, scores, block indices and the library workspace), so the
per-step calls only launch kernels on stable device pointers -- the shape the
C ABI needs for CUDA-graph capture ("prepare-time buffer allocation, stable
data_ptrs", "Eagle3 for M3 MSA path + CUDA graphs compatibility", CUDA-graphs
commit).  PyTorch provides the device memory and streams; all arithmetic runs
in the library's kernels.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (TRTV_BF16, TRTV_F32, geom_of, trtv_draft_attn_p32, trtv_flatten_page_table,
               trtv_msa_proxy_score, trtv_msa_select, trtv_msa_sparse_attn, trtv_msa_topk, trtv_msa_verify,
               trtv_page_table_from_flat,
               trtv_stage_kv, trtv_subpage_view, trtv_verify_dense, trtv_verify_dense_flat,
               trtv_workspace_bytes, trtv_workspace_bytes_flat)
from .workloads import VerifyProblem


class DeviceVerify:
    """Device copies of a problem plus output and workspace buffers."""

    def __init__(self, p: VerifyProblem, device: str = "cuda", num_ctas: int = 0,
                 out_dtype: Optional[str] = None, topk: Optional[int] = None):
        if not torch.cuda.is_available():
            raise RuntimeError("DeviceVerify needs a CUDA device")
        self.p = p
        self.device = torch.device(device)
        self.topk = p.topk if topk is None else topk
        self.geom = geom_of(p, num_ctas=num_ctas)
        od = p.out_dtype if out_dtype is None else out_dtype
        self.out_dtype = TRTV_F32 if od == "f32" else TRTV_BF16
        dev = self.device
        self.q = p.q.to(dev)
        self.pool = p.pool.to(dev)
        self.page_table = p.page_table.to(dev)
        self.kv_lens = p.kv_lens.to(dev)
        B, T, Hq, Hk, D, NP = (p.batch, p.qo_len, p.num_q_heads, p.num_kv_heads, p.head_dim,
                               p.max_pages_per_req)
        self.out = torch.empty(B * T, Hq, D, device=dev,
                               dtype=torch.float32 if self.out_dtype == TRTV_F32 else torch.bfloat16)
        # room for the sparse plan and for a rebuilt flat table
        self.ws_bytes = max(trtv_workspace_bytes(self.geom, max(self.topk, 0)),
                            trtv_workspace_bytes_flat(self.geom))
        if self.ws_bytes == 0:
            raise RuntimeError("geometry rejected by trtv_workspace_bytes")
        # no initial contents needed: each call writes what it reads
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.scores = torch.empty(B, T, Hk, NP, dtype=torch.float32, device=dev)
        k = max(self.topk, 1)
        self.block_idx = torch.empty(B, T, Hk, k, dtype=torch.int32, device=dev)
        self.k_sub = torch.empty(B, 4 * NP, dtype=torch.int32, device=dev)
        self.v_sub = torch.empty(B, 4 * NP, dtype=torch.int32, device=dev)
        self.flat = torch.zeros(B * NP, dtype=torch.int32, device=dev)
        self.indptr = torch.zeros(B + 1, dtype=torch.int32, device=dev)

    # -- single steps -------------------------------------------------------
    def subpage_view(self, stream=None):
        trtv_subpage_view(self.geom, self.page_table, self.kv_lens, self.k_sub, self.v_sub, stream)
        return self.k_sub, self.v_sub

    def dense(self, stream=None):
        trtv_verify_dense(self.geom, self.q, self.pool, self.page_table, self.kv_lens, self.out,
                          self.out_dtype, self.workspace, self.ws_bytes, stream)
        return self.out

    def proxy(self, stream=None):
        trtv_msa_proxy_score(self.geom, self.q, self.pool, self.page_table, self.kv_lens,
                             self.scores, stream)
        return self.scores

    def select(self, scores=None, stream=None):
        trtv_msa_topk(self.geom, self.scores if scores is None else scores, self.kv_lens,
                      self.topk, self.block_idx, stream)
        return self.block_idx

    def select_fused(self, stream=None):
        """Proxy scores and top-k in one call (trtv_msa_select)."""
        trtv_msa_select(self.geom, self.q, self.pool, self.page_table, self.kv_lens, self.topk,
                        self.scores, self.block_idx, self.workspace, self.ws_bytes, stream)
        return self.block_idx

    def msa_verify(self, stream=None):
        """Proxy scores, top-k and sparse attention in one call (trtv_msa_verify)."""
        trtv_msa_verify(self.geom, self.q, self.pool, self.page_table, self.kv_lens, self.topk, self.scores,
                        self.block_idx, self.out, self.out_dtype, self.workspace, self.ws_bytes, stream)
        return self.out

    def sparse(self, block_idx=None, topk: Optional[int] = None, stream=None):
        idx = self.block_idx if block_idx is None else block_idx
        k = self.topk if topk is None else topk
        trtv_msa_sparse_attn(self.geom, self.q, self.pool, self.page_table, self.kv_lens, idx, k,
                             self.out, self.out_dtype, self.workspace, self.ws_bytes, stream)
        return self.out

    def stage(self, k_new, v_new, stream=None):
        """Write the qo_len verify tokens' K and V ([B*T, Hk, D] bf16 CUDA
        tensors) into their cache slots of this problem's pool."""
        trtv_stage_kv(self.geom, k_new, v_new, self.pool, self.page_table, self.kv_lens, stream)
        return self.pool

    def flatten(self, stream=None):
        """Restage the flat (CSR) table and indptr from the page table and the
        current lengths."""
        trtv_flatten_page_table(self.geom, self.page_table, self.kv_lens, self.flat, self.indptr, stream)
        return self.flat, self.indptr

    def table_from_flat(self, flat=None, out=None, stream=None):
        out = torch.empty_like(self.page_table) if out is None else out
        trtv_page_table_from_flat(self.geom, self.flat if flat is None else flat, self.kv_lens, out, stream)
        return out

    def dense_flat(self, flat=None, stream=None):
        """Dense verify taking the flat table (rebuilt on the device)."""
        trtv_verify_dense_flat(self.geom, self.q, self.pool, self.flat if flat is None else flat,
                               self.kv_lens, self.out, self.out_dtype, self.workspace, self.ws_bytes,
                               stream)
        return self.out

    def draft(self, k_sub=None, v_sub=None, stream=None):
        """Attention through the P32 sub-page tables (default: this object's
        k_sub / v_sub, as filled by subpage_view)."""
        trtv_draft_attn_p32(self.geom, self.q, self.pool, self.k_sub if k_sub is None else k_sub,
                            self.v_sub if v_sub is None else v_sub, self.kv_lens, self.out,
                            self.out_dtype, self.workspace, self.ws_bytes, stream)
        return self.out

    def msa(self, stream=None):
        """The MSA sparse verify pass: proxy scores -> per-token top-k -> sparse attention."""
        self.proxy(stream)
        self.select(stream=stream)
        return self.sparse(stream=stream)

    def msa_fused(self, stream=None):
        """The same pass in one call (trtv_msa_verify: fused select building
        the sparse plan, then the sparse attention)."""
        return self.msa_verify(stream)
