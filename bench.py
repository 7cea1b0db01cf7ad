"""Benchmark: multi-token speculative-decoding verify attention on one GB300.

Headline workload ("dense"): batch 64, qo_len 4, kv_len ~ U{1024..8192},
32 query / 4 KV heads, head_dim 128, bf16 K/V in P128 pages read through the
P32 grouped-HND view, bf16 output.  One step = one verify pass of that batch:
the P32 sub-page view (trtv_subpage_view) and the dense ladder attention with
its split-KV merge (trtv_verify_dense).  The other workloads are timed the
same way and printed first, one short JSON line each ("path": msa, fp8, long,
draft), with the KV slot staging and flat-table lines; the headline line is
printed last.

value      query tokens per second (batch * qo_len per step), whole job;
           ms_per_step is the median of repeats of the K-step loop (repeated
           until about a second is timed, so clock samples fall inside it)
e2e        the same through the C ABI with per-step host->device copies of
           q / page table / kv_lens from pinned memory and the output read back
roofline   the dominant call (trtv_verify_dense: the attention kernel and its
           split-combine kernel) timed as the step is, K calls back to back
           with events around the loop (its time is its share of the step),
           against the measured HBM copy bandwidth (also given as a fraction
           of the nominal 8 TB/s); algorithmic bytes = K and V of every
           visible position + Q + O
cpu_baseline  the fp64 oracle on a bounded sample of the same workload

--impl reference runs the fp64 oracle as the reference arm: the sources of
the method are text only, so there is no runnable reference implementation.
Run: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify query-tokens/s and KV HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "query-tokens/s"
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal ("~8 TB/s")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decode_verify_kv_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded by an ncu capture of the current kernel
    sources (profiles/dram_traffic.txt), else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash()
    for line in open(path):
        m = re.match(r"^(\S+)\s+(\S+)\s+([0-9a-f]+)\s+(\d+)", line)
        if m and m.group(1) == kernel and m.group(2) == workload and m.group(3) == want:
            return int(m.group(4))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while running."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        inside = [r for (t, r) in self.rows if t0 <= t <= t1 + 0.15]
        note = None
        if not inside:
            inside = [r for (t, r) in self.rows]
            note = "timed region shorter than the 100 ms sampling period; samples around it"
        mhz, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                maxs.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        out = {"sm_mhz": float(np.median(mhz)) if mhz else None,
               "sm_max_mhz": float(max(maxs)) if maxs else None,
               "reasons": sorted(reasons), "samples": len(mhz)}
        if note:
            out["note"] = note
        return out


# ---------------------------------------------------------------------------
# algorithmic bytes

def dense_bytes(p) -> int:
    elem = p.kv_elem_bytes()
    kv = int(p.kv_lens.sum())
    kv_bytes = kv * p.num_kv_heads * p.head_dim * elem * 2
    q_bytes = p.q.numel() * 2
    o_bytes = p.q.numel() * (4 if p.out_dtype == "f32" else 2)
    return kv_bytes + q_bytes + o_bytes


def proxy_bytes(p) -> int:
    elem = p.kv_elem_bytes()
    k_bytes = int(p.kv_lens.sum()) * p.num_kv_heads * p.head_dim * elem
    return k_bytes + p.q.numel() * 2 + p.batch * p.qo_len * p.num_kv_heads * p.max_pages_per_req * 4


def sparse_bytes(p, idx: np.ndarray):
    """K and V of the visible positions of each unique selected block, per
    (request, KV head), + Q + O + indices.  Also returns the mean unique count."""
    elem = p.kv_elem_bytes()
    lens = p.kv_lens.numpy()
    pos = 0
    uniq = []
    for b in range(p.batch):
        L = int(lens[b])
        npg = (L + 127) // 128
        for h in range(p.num_kv_heads):
            u = np.unique(idx[b, :, h, :])
            u = u[(u >= 0) & (u < npg)]
            uniq.append(len(u))
            pos += int(np.minimum(128, L - 128 * u).sum())
    kv = pos * p.head_dim * elem * 2
    return kv + p.q.numel() * 2 + p.q.numel() * 2 + idx.size * 4, float(np.mean(uniq))


# ---------------------------------------------------------------------------

_CACHE = {}
BATCH = None   # --batch: first requests only (profiling captures), else the full batch


def make(name):
    from speculative_decode_verify_kv_gb300 import workloads as W
    if name not in _CACHE:
        _CACHE[name] = W.make_workload(name, batch=BATCH)
    return _CACHE[name]


def describe(p, name):
    view = ("read through the P32 sub-page tables (drafter attention)" if name == "draft"
            else "P128 pages via P32 grouped-HND view")
    return {"workload": f"{name}: batch {p.batch}, qo_len {p.qo_len}, {p.num_q_heads}/{p.num_kv_heads} "
                        f"heads, head_dim {p.head_dim}, {p.kv_dtype} K/V, {view}, stride "
                        f"{p.slot_stride}" + (f", top-k {p.topk}" if p.topk else ""),
            "batch": p.batch, "qo_len": p.qo_len, "num_q_heads": p.num_q_heads,
            "num_kv_heads": p.num_kv_heads, "head_dim": p.head_dim, "kv_dtype": p.kv_dtype,
            "kv_len_mean": float(p.kv_lens.float().mean()), "kv_len_total": int(p.kv_lens.sum()),
            "pool_slots": p.num_slots, "max_pages_per_req": p.max_pages_per_req,
            "seed": 1000 + ["tiny", "dense", "msa", "fp8", "long", "draft"].index(name)}


def dominant_call(p, name):
    """The call whose kernels dominate a step of workload `name`."""
    return "proxy" if p.topk else ("draft_attn" if name == "draft" else "verify_dense")


def dominant_bytes(p, name) -> int:
    return proxy_bytes(p) if p.topk else dense_bytes(p)


def config_of(p, name, world):
    """The bench line's config (the same dict for both arms)."""
    kv = dominant_bytes(p, name)
    return dict(describe(p, name),
                l2=f"inputs larger than L2: {kv / 2**20:.0f} MiB of KV read per step vs "
                   f"{L2_BYTES / 2**20:.0f} MiB L2, no flush",
                parallelism="replicas" if world > 1 else "single GPU")


def _calls(dv, p, name):
    msa = p.topk > 0
    if msa:
        # proxy, top-k, sparse plan, attention, split combine
        return [("proxy", dv.proxy), ("topk", dv.select), ("sparse", dv.sparse)], 5
    if name == "draft":
        # sub-page view, attention through the P32 tables, split combine
        return [("subpage_view", dv.subpage_view), ("draft_attn", dv.draft)], 3
    return [("subpage_view", dv.subpage_view), ("verify_dense", dv.dense)], 3


def time_path(name, steps, warmup, sampler=None, min_seconds=1.0, max_repeats=20, dist=None):
    """Device-time verify passes of workload `name` (inputs resident in HBM).

    Step: every call of a step goes out back to back (each kernel's
    programmatic dependent launch may overlap the previous one) with events
    only around the K-step loop, which is repeated until `min_seconds` of
    device time (at least once); ms_per_step is the median repeat.  Dominant
    call: the same K-step loop with that call alone (events around the loop),
    so its time is the call's own share of a step; every other call is timed
    alone the same way.  Per-call times of every call inside the step come
    from a third, shorter loop with an event after every call (which keeps
    consecutive calls from overlapping, so these are upper bounds)."""
    import torch
    from speculative_decode_verify_kv_gb300.runtime import DeviceVerify
    p = make(name)
    dv = DeviceVerify(p)
    calls, launches = _calls(dv, p, name)
    dom = dominant_call(p, name)
    dom_f = dict(calls)[dom]
    for _ in range(warmup):
        for _, f in calls:
            f()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def loop(fs):
        a, b = E(), E()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        a.record()
        for _ in range(steps):
            for f in fs:
                f()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    reps = []
    t0 = time.time()
    total = 0.0
    while (total < min_seconds * 1e3 and len(reps) < max_repeats) or not reps:
        ms = loop([f for _, f in calls])
        total += ms
        reps.append(ms / steps)
    t1 = time.time()
    dom_reps = [loop([dom_f]) / steps for _ in range(3)]
    # every call moving KV bytes also timed alone, back to back (median of 3)
    alone = {n: float(np.median([loop([f]) / steps for _ in range(3)])) for n, f in calls if n != dom}
    alone[dom] = float(np.median(dom_reps))
    n_pc = max(10, steps // 8)
    ev = [[E() for _ in range(len(calls) + 1)] for _ in range(n_pc)]
    for k in range(n_pc):
        e = ev[k]
        e[0].record()
        for i, (_, f) in enumerate(calls):
            f()
            e[i + 1].record()
    torch.cuda.synchronize()
    per_call = {n: float(np.mean([ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(n_pc)]))
                for i, (n, _) in enumerate(calls)}
    from speculative_decode_verify_kv_gb300 import trtv_get_device_error
    derr = trtv_get_device_error()
    res = {"p": p, "dv": dv, "ms_per_step": float(np.median(reps)), "repeats": len(reps),
           "timed_s": total / 1e3, "dom": dom, "dom_ms": float(np.median(dom_reps)), "per_call_ms": per_call,
           "alone_ms": alone,
           "t0": t0, "t1": t1, "launches_per_step": launches, "device_error": derr}
    if p.topk:
        idx = dv.block_idx.cpu().numpy()
        sb, umean = sparse_bytes(p, idx)
        res["bytes"] = {"proxy": proxy_bytes(p), "sparse": sb,
                        "topk": p.batch * p.qo_len * p.num_kv_heads * (p.max_pages_per_req * 4 + p.topk * 4)}
        res["unique_blocks_mean"] = umean
    else:
        res["bytes"] = {dom: dense_bytes(p),
                        "subpage_view": p.batch * p.max_pages_per_req * (4 + 32) + p.batch * 4}
    return res


def time_flat(name, steps, warmup):
    """The flat (CSR) page-table entry points on workload `name`: restaging
    the flat table from the lengths, and the dense verify taking the flat
    table (its rebuild kernel + attention + combine) next to the verify on the
    padded table."""
    import torch
    from speculative_decode_verify_kv_gb300.runtime import DeviceVerify
    p = make(name)
    dv = DeviceVerify(p)
    dv.flatten()
    calls = [("flatten", dv.flatten), ("verify_dense_flat", dv.dense_flat), ("verify_dense", dv.dense)]
    out = {}
    for n, f in calls:
        for _ in range(warmup):
            f()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(steps):
            f()
        e.record()
        torch.cuda.synchronize()
        out[n + "_ms"] = s.elapsed_time(e) / steps
    out["launches"] = {"flatten": 1, "verify_dense_flat": 3, "verify_dense": 2}
    del dv
    torch.cuda.empty_cache()
    return out


def time_msa_fused(name, steps, warmup):
    """The MSA pass as one call (trtv_msa_verify: the top-k fused into the
    proxy kernel, which also builds the sparse plan, then the attention): the
    step time, and the select call (trtv_msa_select) on its own."""
    import torch
    from speculative_decode_verify_kv_gb300.runtime import DeviceVerify
    p = make(name)
    dv = DeviceVerify(p)
    out = {}
    for label, calls in (("step", [dv.msa_verify]), ("select", [dv.select_fused])):
        for _ in range(warmup):
            for f in calls:
                f()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(steps):
            for f in calls:
                f()
        e.record()
        torch.cuda.synchronize()
        out[label + "_ms"] = s.elapsed_time(e) / steps
    out["launches_per_step"] = 4   # counter zeroing, proxy with fused top-k and plan, attention, combine
    from speculative_decode_verify_kv_gb300 import trtv_get_device_error
    out["device_error"] = trtv_get_device_error()
    del dv
    torch.cuda.empty_cache()
    return out


def time_stage(name, steps, warmup):
    """trtv_stage_kv on workload `name`: the qo_len new tokens' K and V of
    every request written into their cache slots (device-resident inputs)."""
    import torch
    from speculative_decode_verify_kv_gb300.runtime import DeviceVerify
    p = make(name)
    dv = DeviceVerify(p)
    g = torch.Generator().manual_seed(99)
    shape = (p.batch * p.qo_len, p.num_kv_heads, p.head_dim)
    k_new = torch.randn(shape, generator=g).to(torch.bfloat16).cuda()
    v_new = torch.randn(shape, generator=g).to(torch.bfloat16).cuda()
    for _ in range(warmup):
        dv.stage(k_new, v_new)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        dv.stage(k_new, v_new)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    n = k_new.numel() * 2
    nbytes = n * 2 + n * p.kv_elem_bytes() + p.batch * 4 * 3
    del dv
    torch.cuda.empty_cache()
    return {"ms": ms, "bytes": int(nbytes), "gbs": nbytes / (ms / 1e3) / 1e9, "launches_per_call": 1}


def time_e2e(name, steps, warmup):
    """Same step through the C ABI with host buffers: per step, H2D of q,
    page table and kv_lens from pinned memory, the kernels, D2H of the output.

    Pipelined (the reported value): two sets of device buffers (one shared KV
    pool); step i's copies run on a copy stream -- its inputs while step i - 1
    computes, its output while step i + 1 computes -- and every step's copies
    and kernels lie inside the timed region (events around the whole loop,
    the compute stream joining the copy stream at the end).  Serial: the same
    copies and kernels in order on one stream (reported beside it)."""
    import torch
    from speculative_decode_verify_kv_gb300.runtime import DeviceVerify
    p = make(name)
    dvs = [DeviceVerify(p), DeviceVerify(p)]
    dvs[1].pool = dvs[0].pool  # one resident KV pool
    torch.cuda.empty_cache()
    hq = p.q.pin_memory()
    hpt = p.page_table.pin_memory()
    hl = p.kv_lens.pin_memory()
    houts = [torch.empty(dvs[0].out.shape, dtype=dvs[0].out.dtype).pin_memory() for _ in range(2)]
    msa = p.topk > 0
    comp = torch.cuda.current_stream()
    cs = torch.cuda.Stream()
    E = lambda: torch.cuda.Event()  # noqa: E731
    ev_in = [E(), E()]
    ev_done = [E(), E()]
    for e in ev_done:
        e.record(comp)

    def h2d(k, stream):
        d = dvs[k]
        with torch.cuda.stream(stream):
            stream.wait_event(ev_done[k])  # the previous step on these buffers has finished
            d.q.copy_(hq, non_blocking=True)
            d.page_table.copy_(hpt, non_blocking=True)
            d.kv_lens.copy_(hl, non_blocking=True)
            ev_in[k].record(stream)

    def kernels(k):
        d = dvs[k]
        comp.wait_event(ev_in[k])
        if msa:
            d.msa()
        else:
            d.subpage_view()
            d.dense()
        ev_done[k].record(comp)

    def d2h(k, stream):
        with torch.cuda.stream(stream):
            stream.wait_event(ev_done[k])
            houts[k].copy_(dvs[k].out, non_blocking=True)

    def pipelined(n):
        h2d(0, cs)
        for i in range(n):
            k = i & 1
            kernels(k)
            if i + 1 < n:
                h2d(k ^ 1, cs)
            d2h(k, cs)
        comp.wait_stream(cs)

    def serial(n):
        for i in range(n):
            h2d(0, comp)
            kernels(0)
            d2h(0, comp)

    out = {}
    for label, run in (("pipelined", pipelined), ("serial", serial)):
        run(warmup)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(comp)
        cs.wait_stream(comp)
        run(steps)
        e.record(comp)
        torch.cuda.synchronize()
        out[label] = s.elapsed_time(e) / steps
    ms = out["pipelined"]
    h2d_b = hq.numel() * hq.element_size() + hpt.numel() * 4 + hl.numel() * 4
    d2h_b = houts[0].numel() * houts[0].element_size()
    res = {"value": p.batch * p.qo_len / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
           "h2d_bytes_per_step": int(h2d_b), "d2h_bytes_per_step": int(d2h_b),
           "copies": "copy stream, double-buffered, overlapping the neighbouring steps' kernels",
           "serial_value": p.batch * p.qo_len / (out["serial"] / 1e3), "serial_ms_per_step": out["serial"]}
    del dvs
    torch.cuda.empty_cache()
    return res


def cpu_baseline(name, budget_s=12.0):
    """The fp64 oracle, as it stands, on a bounded sample of the workload's
    requests (same pool); throughput scaled to query tokens/s."""
    import oracle
    p = make(name)
    Tq = p.qo_len
    import torch
    n = 1
    spent = 0.0
    while True:
        reqs = list(range(min(n, p.batch)))
        rows = torch.cat([torch.arange(b * Tq, (b + 1) * Tq) for b in reqs])
        x = oracle.Inputs(p, q=p.q[rows], page_table=p.page_table[reqs].contiguous(),
                          kv_lens=p.kv_lens[reqs].contiguous(), batch=len(reqs))
        t0 = time.perf_counter()
        if p.topk:
            s, _ = oracle.proxy_score(x)
            idx, _ = oracle.topk(x, s, p.topk)
            oracle.sparse_attn(x, idx)
        else:
            oracle.subpage_view(x)
            oracle.verify_dense(x)
        dt = time.perf_counter() - t0
        spent += dt
        if dt > budget_s / 4 or len(reqs) == p.batch or spent > budget_s:
            break
        n *= 2
    return {"value": len(reqs) * Tq / dt, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"first {len(reqs)} of {p.batch} requests of the {name} workload "
                      f"({int(p.kv_lens[:len(reqs)].sum())} KV positions), one pass, {dt:.2f} s"}


def max_over_ranks(x: float, dist=None, device="cuda") -> float:
    """The largest of every rank's x: the job's step time is its slowest
    replica's (each rank runs the whole workload on its own GPU; no data
    crosses ranks)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job query tokens per second: every replica's tokens over the
    slowest replica's step time."""
    return tokens_per_rank * world / (ms / 1e3)


def run_reference(args):
    """Reference arm: the fp64 oracle on the host cores, each step a bounded
    sample (4 requests, rotating) of the same workload."""
    import torch
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    p = make(args.workload)
    Tq = p.qo_len
    per = min(4, p.batch)

    def step(k):
        reqs = [(k * per + i) % p.batch for i in range(per)]
        rows = torch.cat([torch.arange(b * Tq, (b + 1) * Tq) for b in reqs])
        x = oracle.Inputs(p, q=p.q[rows], page_table=p.page_table[reqs].contiguous(),
                          kv_lens=p.kv_lens[reqs].contiguous(), batch=len(reqs))
        if p.topk:
            s, _ = oracle.proxy_score(x)
            idx, _ = oracle.topk(x, s, p.topk)
            oracle.sparse_attn(x, idx)
        else:
            oracle.subpage_view(x)
            oracle.verify_dense(x)

    for k in range(args.warmup):
        step(k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(args.warmup + k)
    dt = time.perf_counter() - t0
    value = per * Tq * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(p, args.workload, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{per} requests per step of the {args.workload} workload"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="dense", choices=["dense", "msa", "fp8", "long", "draft"])
    ap.add_argument("--paths", default="msa,fp8,long,draft",
                    help="extra workloads timed alongside (comma list, or none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="keep only the first requests of each workload (small profiling case)")
    args = ap.parse_args()
    global BATCH
    BATCH = args.batch
    if args.impl == "reference":
        run_reference(args)
        return
    if args.warmup < 3:
        args.warmup = 3

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import speculative_decode_verify_kv_gb300 as T
    from speculative_decode_verify_kv_gb300 import _build
    _build.build()
    T.load()
    T.trtv_get_device_error()

    sampler = ClockSampler(local)
    peak, peak_kind = peaks()

    def sig(x, n=4):
        return float(f"{x:.{n}g}")

    def path_line(name, r):
        """One short JSON line per workload: step, per-call and dominant times."""
        pe = r["p"]
        step_bytes = sum(r["bytes"].values())
        gbs = step_bytes / (r["ms_per_step"] / 1e3) / 1e9
        calls = {}
        for n, b in r["bytes"].items():
            ms_c = r["per_call_ms"][n]
            g = b / (ms_c / 1e3) / 1e9
            calls[n] = [sig(ms_c * 1e3), sig(g), sig(g / peak, 3)]
        dg = r["bytes"][r["dom"]] / (r["dom_ms"] / 1e3) / 1e9
        alone = {}
        for n, b in r["bytes"].items():
            if b < 1e8:  # the KV-streaming calls only
                continue
            ms_c = r["alone_ms"][n]
            g = b / (ms_c / 1e3) / 1e9
            alone[n] = [sig(ms_c * 1e3), sig(g), sig(g / peak, 3), sig(g / NOMINAL_HBM_GBS, 3)]
        return {"path": name, "workload": describe(pe, name)["workload"],
                "value": sig(pe.batch * pe.qo_len / (r["ms_per_step"] / 1e3)), "unit": UNIT,
                "ms_per_step": sig(r["ms_per_step"]), "repeats": r["repeats"],
                "step_gbs": sig(gbs), "step_frac_of_measured": sig(gbs / peak, 3),
                "step_frac_of_8tbs": sig(gbs / NOMINAL_HBM_GBS, 3),
                "dominant": {"call": r["dom"], "us_alone": sig(r["dom_ms"] * 1e3), "gbs": sig(dg),
                             "frac_of_measured": sig(dg / peak, 3), "frac_of_8tbs": sig(dg / NOMINAL_HBM_GBS, 3)},
                "calls_us_gbs_frac": calls,
                "calls_alone_us_gbs_frac_of_measured_frac_of_8tbs": alone, "device_error": r["device_error"],
                "gpu_launches_per_step": r["launches_per_step"]}

    # ---- other workloads first (one short line each), then the headline
    summary = {}
    for extra in [w for w in args.paths.split(",") if w and w not in (args.workload, "none")]:
        r = time_path(extra, max(10, args.steps // 8), args.warmup, min_seconds=0.3, dist=dist)
        pl = path_line(extra, r)
        if "unique_blocks_mean" in r:
            pl["unique_blocks_mean"] = sig(r["unique_blocks_mean"])
        if r["p"].topk:
            f = time_msa_fused(extra, max(10, args.steps // 8), args.warmup)
            pl["fused_select"] = {"step_us": sig(f["step_ms"] * 1e3), "select_us": sig(f["select_ms"] * 1e3),
                                  "device_error": f["device_error"]}
        else:
            st = time_stage(extra, max(10, args.steps // 8), args.warmup)
            pl["stage_kv"] = {"us": sig(st["ms"] * 1e3), "bytes": st["bytes"], "gbs": sig(st["gbs"])}
        summary[extra] = {"value": pl["value"], "ms_per_step": pl["ms_per_step"],
                          "dominant_frac_of_measured": pl["dominant"]["frac_of_measured"]}
        if rank == 0:
            print(json.dumps(pl), flush=True)
        del r
        _CACHE.pop(extra, None)
        torch.cuda.empty_cache()

    if dist:
        dist.barrier()
    head = time_path(args.workload, args.steps, args.warmup, sampler, dist=dist)
    sampler.stop()
    clocks = sampler.summary(head["t0"], head["t1"])
    ms = max_over_ranks(head["ms_per_step"], dist)
    p = head["p"]
    qtok = p.batch * p.qo_len
    value = job_value(qtok, world, ms)
    if rank == 0:
        print(json.dumps(path_line(args.workload, head)), flush=True)

    dom = head["dom"]
    dom_ms = head["dom_ms"]
    dom_bytes = head["bytes"][dom]
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    step_bytes = sum(head["bytes"].values())
    kernel_name = ("proxy_umma_kernel" if p.topk else
                   "attn_kernel; the timed call also holds the split-combine kernel")
    roofline = {"bound": "hbm", "achieved": sig(achieved), "peak": peak, "unit": "GB/s",
                "frac": sig(achieved / peak, 4), "traffic": ncu_traffic(dom, args.workload),
                "kernel": f"{dom} ({kernel_name})", "peak_kind": f"of {peak_kind}",
                "algorithmic_bytes": dom_bytes, "launch_ms": sig(dom_ms),
                "frac_of_nominal_8tbs": sig(achieved / NOMINAL_HBM_GBS, 4)}

    stage = time_stage(args.workload, max(10, args.steps // 8), args.warmup)
    if rank == 0:
        print(json.dumps({"aux": "stage_kv", "workload": args.workload, "us": sig(stage["ms"] * 1e3),
                          "bytes": stage["bytes"], "gbs": sig(stage["gbs"]), "launches_per_call": 1}), flush=True)
    if not p.topk:
        flat = time_flat(args.workload, max(10, args.steps // 8), args.warmup)
        if rank == 0:
            print(json.dumps({"aux": "flat_table", "workload": args.workload,
                              "flatten_us": sig(flat["flatten_ms"] * 1e3),
                              "verify_dense_flat_us": sig(flat["verify_dense_flat_ms"] * 1e3),
                              "verify_dense_us": sig(flat["verify_dense_ms"] * 1e3),
                              "launches": flat["launches"]}), flush=True)

    e2e = None if args.no_e2e else time_e2e(args.workload, max(10, args.steps // 4), args.warmup)
    if dist and e2e:
        e2e["value"] = job_value(qtok, world, max_over_ranks(e2e["ms_per_step"], dist))
        e2e["serial_value"] = job_value(qtok, world, max_over_ranks(e2e["serial_ms_per_step"], dist))

    gbs = step_bytes / (ms / 1e3) / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "repeats": head["repeats"],
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": p.kv_dtype.replace("fp8_e4m3", "fp8e4m3"),
            "data": "synthetic", "config": config_of(p, args.workload, world),
            "kv_hbm_gbs": sig(gbs), "kv_hbm_pct_of_measured_peak": sig(100 * gbs / peak),
            "kv_hbm_pct_of_nominal_8tbs": sig(100 * gbs / NOMINAL_HBM_GBS),
            "per_call_ms": {k: sig(v) for k, v in head["per_call_ms"].items()}, "roofline": roofline,
            "e2e": ({k: (sig(e2e[k]) if k.endswith("value") else e2e[k])
                     for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step", "copies",
                               "serial_value")}
                    if e2e else None),
            "gpu_launches": head["launches_per_step"] * args.steps * head["repeats"],
            "clocks": clocks, "device_error": head["device_error"], "paths": summary}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
