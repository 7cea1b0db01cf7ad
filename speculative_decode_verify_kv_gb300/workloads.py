"""Seeded synthetic inputs for verify attention over a paged KV cache.

This module only draws random numbers and lays out the caller-visible
buffers (query rows, page pool, page table, per-request KV lengths).  It holds
none of the method's arithmetic: no attention, no scoring, no selection and no
sub-page address mapping.  Both the CUDA path and the fp64 oracle consume the
same host tensors produced here.

Pool storage (the only layout fact used here): the pool is an array of page
buffers, each one ``[4 token groups, kv_heads, 32, head_dim]`` elements; a
slot owns ``slot_stride`` consecutive buffers, of which the first is this
layer's K page and the second its V page ("slot s's K at s * stride and its V
at s * stride + 1", TensorRT-LLM PR #18066, MiniMaxM3DraftKVCacheView commit).
Buffers of slots no request uses are left zero; buffers of used slots (and of
slot 0, which padded page-table entries address) are filled with N(0, 1).

Workloads (sizes and distributions of the five verify configurations):

====  ==================================================================
name  shape
====  ==================================================================
tiny  B=2, T=4, kv_len {100, 257}, Hq=8, Hk=2, D=64, 8-slot pool, fp32 out
dense B=64, T=4, kv_len ~ U{1024..8192}, Hq=32, Hk=4, D=128, 12288-slot pool
msa   B=32, T=4, kv_len ~ U{16384..65536}, Hq=64, Hk=4, D=128, top-k 16
fp8   B=256, T=4, kv_len = clip(round(4096 e^N(0,1)), 256, 32768), FP8 K/V
long  B=8, T=8, kv_len 131072, Hq=64, Hk=4, D=128, 5% of K blocks +2.0, k=32
====  ==================================================================
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import torch

PAGE = 128          # tokens per physical page
SUBPAGE = 32        # tokens per sub-page of the grouped-HND view
GROUPS = PAGE // SUBPAGE

BF16 = "bf16"
FP8 = "fp8_e4m3"


@dataclass
class VerifyProblem:
    """One batch of verify inputs, all tensors on the host (CPU)."""
    name: str
    batch: int
    qo_len: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    max_pages_per_req: int
    num_slots: int
    slot_stride: int
    kv_dtype: str
    sm_scale: float
    k_scale: float
    v_scale: float
    topk: int
    out_dtype: str
    q: torch.Tensor            # bf16 [B*T, Hq, D]
    pool: torch.Tensor         # bf16 or uint8 [num_slots*stride, 4, Hk, 32, D]
    page_table: torch.Tensor   # int32 [B, max_pages_per_req]
    kv_lens: torch.Tensor      # int32 [B]
    shifted_slots: Optional[torch.Tensor] = None  # slots whose K got +shift
    notes: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == FP8 else 2

    def pages_per_req(self) -> torch.Tensor:
        return (self.kv_lens.to(torch.int64) + PAGE - 1) // PAGE

    def with_(self, **kw) -> "VerifyProblem":
        return replace(self, **kw)


def _randn_bf16(n: int, gen: torch.Generator, chunk: int = 1 << 24) -> torch.Tensor:
    out = torch.empty(n, dtype=torch.bfloat16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return out


def _randn_f32(n: int, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(n, generator=gen, dtype=torch.float32)


def make_problem(*, name: str = "custom", kv_lens: Sequence[int], qo_len: int,
                 num_q_heads: int, num_kv_heads: int, head_dim: int,
                 max_pages_per_req: Optional[int] = None, num_slots: Optional[int] = None,
                 slot_stride: int = 2, kv_dtype: str = BF16, sm_scale: Optional[float] = None,
                 topk: int = 0, out_dtype: str = "bf16", seed: int = 0,
                 slack_slots: int = 0, fill_unused_with=None,
                 shift_fraction: float = 0.0, shift_value: float = 0.0,
                 other_buffers=None) -> VerifyProblem:
    """Build one seeded problem.

    Page ids are a random permutation of the pool's slots handed to requests in
    order; unused page-table entries are 0.  ``fill_unused_with`` (a float, e.g.
    ``float('nan')``) fills every buffer of slots no request uses.
    ``shift_fraction`` of each request's pages get ``shift_value`` added to all
    K elements of that slot (the long-context workload's distinct winners).
    ``other_buffers`` (a float): buffers 2.. of every used slot -- the pages of
    other layers in a pool with a wider slot stride -- hold that value instead
    of random draws (only this layer's K and V pages are drawn).
    """
    B = len(kv_lens)
    lens = torch.tensor(list(kv_lens), dtype=torch.int32)
    pages = [(int(L) + PAGE - 1) // PAGE for L in kv_lens]
    if max_pages_per_req is None:
        max_pages_per_req = max(1, max(pages))
    total = sum(pages)
    if num_slots is None:
        num_slots = total + slack_slots
    assert num_slots >= total, "pool too small for the requests"
    gen = torch.Generator().manual_seed(seed)
    # sub-streams drawn in a fixed order: page permutation, q, pool, shifts
    perm = torch.randperm(num_slots, generator=gen).to(torch.int32)
    pt = torch.zeros(B, max_pages_per_req, dtype=torch.int32)
    cur = 0
    for b, n in enumerate(pages):
        n_eff = min(n, max_pages_per_req)
        pt[b, :n_eff] = perm[cur:cur + n_eff]
        cur += n
    Hq, Hk, D, T = num_q_heads, num_kv_heads, head_dim, qo_len
    q = _randn_bf16(B * T * Hq * D, gen).view(B * T, Hq, D)
    buf_elems = GROUPS * Hk * SUBPAGE * D
    used = torch.unique(torch.cat([perm[:total].to(torch.int64), torch.zeros(1, dtype=torch.int64)]))
    n_used = used.numel()
    n_draw = slot_stride if other_buffers is None else min(2, slot_stride)
    n_vals = n_used * n_draw * buf_elems
    vals = _randn_f32(n_vals, gen) if kv_dtype == FP8 else _randn_bf16(n_vals, gen)
    vals = vals.view(n_used, n_draw, buf_elems)
    shifted = None
    if shift_fraction > 0.0:
        pick = []
        for b, n in enumerate(pages):
            m = max(1, int(round(shift_fraction * n)))
            sel = torch.randperm(n, generator=gen)[:m]
            pick.append(pt[b, sel].to(torch.int64))
        shifted = torch.unique(torch.cat(pick))
        pos = torch.searchsorted(used, shifted)
        # buffer 0 of a slot is this layer's K page
        vals[pos, 0] = (vals[pos, 0].to(torch.float32) + shift_value).to(vals.dtype)
    k_scale = v_scale = 1.0
    if kv_dtype == FP8:
        amax = float(vals.abs().max())
        scale = amax / 448.0
        vals = (vals / scale).to(torch.float8_e4m3fn).view(torch.uint8)
        k_scale = v_scale = scale
        pool_dtype = torch.uint8
    else:
        pool_dtype = torch.bfloat16
    pool = torch.zeros(num_slots, slot_stride, buf_elems, dtype=pool_dtype)
    def stored(x):
        if kv_dtype == FP8:
            return int(torch.tensor([x], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).item())
        return x
    if fill_unused_with is not None:
        pool.fill_(stored(fill_unused_with))
    if n_draw < slot_stride:
        pool[used, n_draw:] = stored(other_buffers)
    pool[used, :n_draw] = vals
    pool = pool.view(num_slots * slot_stride, GROUPS, Hk, SUBPAGE, D)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    return VerifyProblem(name=name, batch=B, qo_len=T, num_q_heads=Hq, num_kv_heads=Hk,
                         head_dim=D, max_pages_per_req=max_pages_per_req, num_slots=num_slots,
                         slot_stride=slot_stride, kv_dtype=kv_dtype, sm_scale=float(sm_scale),
                         k_scale=float(k_scale), v_scale=float(v_scale), topk=topk,
                         out_dtype=out_dtype, q=q, pool=pool, page_table=pt, kv_lens=lens,
                         shifted_slots=shifted)


def _uniform_lens(gen: torch.Generator, B: int, lo: int, hi: int) -> list:
    return torch.randint(lo, hi + 1, (B,), generator=gen).tolist()


def _lognormal_lens(gen: torch.Generator, B: int, median: float, sigma: float,
                    lo: int, hi: int) -> list:
    z = torch.randn(B, generator=gen, dtype=torch.float64)
    L = torch.round(median * torch.exp(sigma * z)).clamp(lo, hi).to(torch.int64)
    return L.tolist()


WORKLOADS = ("tiny", "dense", "msa", "fp8", "long", "draft")


def make_workload(name: str, *, batch: Optional[int] = None, seed: Optional[int] = None,
                  **overrides) -> VerifyProblem:
    """The verify workloads by name (the five configurations plus the drafter's
    P32 decode step, "draft"); ``batch`` keeps the first requests only
    (same lens, same draws for them) so a test can run a reduced copy."""
    idx = WORKLOADS.index(name)
    s = 1000 + idx if seed is None else seed
    lgen = torch.Generator().manual_seed(s + 7919)   # lens sub-stream
    if name == "tiny":
        kw = dict(kv_lens=[100, 257], qo_len=4, num_q_heads=8, num_kv_heads=2, head_dim=64,
                  num_slots=8, slot_stride=2, out_dtype="f32")
    elif name == "dense":
        kw = dict(kv_lens=_uniform_lens(lgen, 64, 1024, 8192), qo_len=4, num_q_heads=32,
                  num_kv_heads=4, head_dim=128, max_pages_per_req=64, num_slots=12288)
    elif name == "msa":
        kw = dict(kv_lens=_uniform_lens(lgen, 32, 16384, 65536), qo_len=4, num_q_heads=64,
                  num_kv_heads=4, head_dim=128, max_pages_per_req=512, slack_slots=1024, topk=16)
    elif name == "fp8":
        kw = dict(kv_lens=_lognormal_lens(lgen, 256, 4096.0, 1.0, 256, 32768), qo_len=4,
                  num_q_heads=32, num_kv_heads=4, head_dim=128, max_pages_per_req=256,
                  slack_slots=1024, kv_dtype=FP8)
    elif name == "long":
        kw = dict(kv_lens=[131072] * 8, qo_len=8, num_q_heads=64, num_kv_heads=4, head_dim=128,
                  max_pages_per_req=1024, slack_slots=1024, topk=32, shift_fraction=0.05,
                  shift_value=2.0)
    elif name == "draft":
        # the drafter's decode step over its FP8 layer, read through the P32
        # tables; slots hold eight page buffers (layer-local stride 8)
        kw = dict(kv_lens=_uniform_lens(lgen, 64, 1024, 8192), qo_len=1, num_q_heads=32,
                  num_kv_heads=4, head_dim=128, max_pages_per_req=64, slack_slots=1024,
                  slot_stride=8, kv_dtype=FP8, other_buffers=0.0)
    else:
        raise KeyError(name)
    if batch is not None:
        kw["kv_lens"] = kw["kv_lens"][:batch]
        if "num_slots" in kw and name != "tiny":
            kw.pop("num_slots")
            kw["slack_slots"] = 64
    kw.update(overrides)
    return make_problem(name=name, seed=s, **kw)
