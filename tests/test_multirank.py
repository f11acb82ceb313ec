"""bench.py's multi-process path on the CPU: two gloo ranks (127.0.0.1).

The decode path does not shard across GPUs here (replicas only); what runs
with N > 1 is the host logic around the replicas: rank/world parsing, the
barrier, the max-over-ranks of the timings, and rank 0 alone printing the
reference line.
"""

import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        bench.barrier(w)
        mx = bench.max_over_ranks(10.0 + r, w)
        buf = io.StringIO()

        class A:
            steps, warmup = 2, 1
        orig = bench.run_oracle
        bench.run_oracle = lambda budget_s, max_steps, n_pos, warmup: {"steps": max_steps,
                                                                       "seconds": 0.5}
        with redirect_stdout(buf):
            bench.run_reference(A, r, w, local)
        bench.run_oracle = orig
        q.put((r, (r, w, local), mx, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_max_and_reference_printing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, env0, mx0, out0), (r1, env1, mx1, out1) = res
    assert env0 == (0, 2, 0) and env1 == (1, 2, 1)
    assert mx0 == mx1 == 11.0
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["unit"] == "GB/s"
    assert out1 == ""          # only rank 0 prints
