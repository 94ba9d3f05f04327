"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2).

Each rank runs an independent batch (weak scaling); the only cross-rank
operations are the barrier and the max over ranks of the step time.  The
reference arm runs on rank 0 only.
"""

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, loc = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.5 + rank, w)  # rank 1 is the slow one
    out = {"rank": r, "world": w, "local": loc, "slowest": slowest}
    if r != 0:
        out["reference_line"] = bench.run_reference(None, r, w)
    q.put(out)
    torch.distributed.destroy_process_group()


def test_two_rank_gloo_max_and_reference_rank0_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort(key=lambda d: d["rank"])
    assert [d["world"] for d in res] == [2, 2]
    assert all(d["slowest"] == 2.5 for d in res)
    assert res[1]["reference_line"] is None  # non-zero ranks print nothing and do no work


def test_bench_parses_its_default_arguments(monkeypatch):
    import sys
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.gpus == 1 and a.steps >= 1 and a.warmup >= 3 and a.impl == "ours"
    assert set(bench.STUDIES) >= {"formats", "stack", "gemv_shapes"}
