"""The N > 1 path of bench.py on CPU: world size 2 over gloo (127.0.0.1).

Each rank runs an independent replica (the decode step has no cross-request
exchange), so the only collectives are the timing reductions: the per-step
time is the max over ranks, and only rank 0 prints the reference line.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w, local = bench.dist_env()
    bench.dist_init(w, "gloo")
    got = bench.reduce_max(10.0 * (rank + 1), w)
    bench.barrier(w)
    import io
    import contextlib
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(bench.main.__globals__["argparse"].Namespace(
            gpus=w, steps=3, warmup=3, workload="tiny", budget=None, pages=None), r, w)
    q.put((rank, got, buf.getvalue()))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_timing_and_rank0_reference_line():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [20.0, 20.0]          # max over ranks on every rank
    assert '"impl": "reference"' in res[0][2]            # rank 0 prints the reference arm
    assert res[1][2] == ""                               # other ranks print nothing
