"""The N > 1 path of bench.py on CPU: two gloo ranks (replicas only -- no
collective on the data path, only the barrier and the timing reductions)."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_setup(use_cuda=False)
    bench.barrier(w, use_cuda=False)
    mx = bench.max_over_ranks(1.5 + r, w, use_cuda=False)
    sm = bench.sum_over_ranks(10.0 * (r + 1), w, use_cuda=False)

    class A:
        workload, T, layers, steps, warmup = "tiny", None, None, 1, 0
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A, r, w, 0)
    dist.destroy_process_group()
    q.put((r, w, mx, sm, buf.getvalue()))


def test_two_gloo_ranks():
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
    (r0, w0, mx0, sm0, out0), (r1, w1, mx1, sm1, out1) = res
    assert (w0, w1) == (2, 2)
    assert mx0 == mx1 == 2.5      # max over ranks of the per-rank times
    assert sm0 == sm1 == 30.0     # whole-job units = sum over ranks
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert out1.strip() == ""     # only rank 0 prints; rank 1 exits without work
