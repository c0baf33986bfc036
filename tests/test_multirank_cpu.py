"""The benchmark's multi-rank path on the CPU: two processes over gloo (one process
per GPU is the contract on a GPU node; here the ranks only exercise the host logic).
Each rank runs the same setup, barrier and max/sum reductions that turn per-rank
timings into the JSON line's ms_per_step (max over ranks) and value (sum over
ranks), and the reference arm's non-zero ranks leave without doing any work."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="gloo ranks on CPU hosts; GPU nodes use NCCL")


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    w, r, _, pg = bench.dist_setup(None)
    bench.barrier(pg)
    mx = bench.max_over_ranks(pg, 1.5 + r)
    sm = bench.sum_over_ranks(pg, 1.5 + r)
    bench.barrier(pg)
    out = (r, w, mx, sm)
    if r != 0:
        # the reference arm: ranks other than 0 return at once, before any oracle work
        class A:
            lam_a, ref_units, steps, warmup = 40.0, 1, 1, 3
        bench.dist_setup = lambda args: (w, r, r, pg)  # the group this process already joined
        out = out + (bench.run_reference(A()),)
    q.put(out)
    pg.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_bench_line():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in procs)
    assert res[0] == (0, 2, 2.5, 4.0)
    assert res[1] == (1, 2, 2.5, 4.0, 0)
