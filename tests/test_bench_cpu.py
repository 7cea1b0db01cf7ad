"""The bench's host logic on the CPU: algorithmic byte counts (hand-worked on
the tiny workload and brute-forced for the sparse count), the replica
arithmetic, and the reference arm's JSON line."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decode_verify_kv_gb300 import workloads as W  # noqa: E402


def test_dense_bytes_tiny_by_hand():
    # kv_len {100, 257}: 357 positions x 2 KV heads x 64 dims x 2 B x (K and V)
    # + Q 2*4 rows x 8 heads x 64 x 2 B + fp32 O of the same shape
    p = W.make_workload("tiny")
    assert bench.dense_bytes(p) == 357 * 2 * 64 * 2 * 2 + 2 * 4 * 8 * 64 * 2 + 2 * 4 * 8 * 64 * 4


def test_sparse_bytes_brute_force():
    p = W.make_problem(kv_lens=[300, 1000, 129], qo_len=4, num_q_heads=8, num_kv_heads=2, head_dim=64,
                       seed=9, topk=3)
    rng = np.random.default_rng(9)
    idx = rng.integers(-1, 9, size=(p.batch, p.qo_len, p.num_kv_heads, 3)).astype(np.int32)
    got, mean_unique = bench.sparse_bytes(p, idx)
    pos = 0
    uniq = []
    for b in range(p.batch):
        L = int(p.kv_lens[b])
        for h in range(p.num_kv_heads):
            blocks = {int(v) for v in idx[b, :, h, :].ravel() if 0 <= v and v * 128 < L}
            uniq.append(len(blocks))
            for v in blocks:                       # every position of the block below kv_len
                pos += sum(1 for q in range(v * 128, v * 128 + 128) if q < L)
    want = pos * 64 * 2 * 2 + 2 * p.q.numel() * 2 + idx.size * 4
    assert got == want
    assert abs(mean_unique - float(np.mean(uniq))) < 1e-12


def test_replica_arithmetic_single_rank():
    assert bench.max_over_ranks(0.25) == 0.25
    assert abs(bench.job_value(256, 1, 0.1) - 2.56e6) < 1e-6


def test_reference_arm_line():
    args = type("A", (), {"workload": "tiny", "warmup": 1, "steps": 2, "gpus": 1})()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    line = json.loads(buf.getvalue())
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "dtype", "config", "cpu_baseline", "e2e", "impl"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    # the same config dict as the GPU arm prints for this workload
    assert line["config"] == bench.config_of(bench.make("tiny"), "tiny", 1)
