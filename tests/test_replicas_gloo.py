"""The N > 1 path on the CPU: two gloo ranks.  Verify attention has no
exchange step, so the only cross-rank logic is the bench's timing: the step
time is the slowest replica's and the value counts every replica's tokens;
the reference arm prints on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(0.100 + 0.050 * rank, dist, device="cpu")
    value = bench.job_value(256, world, ms)
    buf = io.StringIO()
    with redirect_stdout(buf):
        if rank != 0:   # other ranks leave the reference arm without work
            bench.run_reference(type("A", (), {"workload": "tiny", "warmup": 0, "steps": 1, "gpus": world})())
    out.put((rank, ms, value, buf.getvalue()))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    for rank, ms, value, printed in res:
        assert abs(ms - 0.150) < 1e-12                      # both ranks see the max
        assert abs(value - 256 * 2 / 0.150e-3) < 1e-6       # tokens of every replica
        assert printed == ""
