"""The N > 1 host path of bench.py on CPU: two gloo ranks.

Every rank runs its own replica of the workload (no collective in the data
path); ranks only meet at the barriers around the timed loop and in the
max-over-ranks reduction of the timings.  This checks that reduction, the
barrier, and that only rank 0 runs the CPU reference arm.
"""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
world, rank, local = bench.dist_env()
bench.init_dist(world, "gloo")
bench.barrier(world)
vals = bench.max_over_ranks([float(rank + 1), float(10 - rank), 0.5], world)
bench.barrier(world)
out = {{"rank": rank, "world": world, "max": vals}}
print(json.dumps(out))
dist.destroy_process_group()
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _launch(code, world=2, timeout=120):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, WORLD_SIZE=str(world), RANK=str(rank),
                   LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env,
                                      stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        assert p.returncode == 0, e[-2000:]
        outs.append(o)
    return outs


def test_two_rank_max_reduction_and_barrier():
    import json
    outs = _launch(WORKER.format(root=ROOT))
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o in outs),
                 key=lambda r: r["rank"])
    assert [r["rank"] for r in res] == [0, 1]
    for r in res:
        assert r["world"] == 2
        assert r["max"] == [2.0, 10.0, 0.5]


def test_reference_arm_runs_on_rank_zero_only():
    code = r"""
import os, sys
sys.path.insert(0, {root!r})
import bench
class A: steps = 1; warmup = 3
bench.run_reference(A())
""".format(root=ROOT)
    port = _free_port()
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
               CUDA_VISIBLE_DEVICES="")
    p = subprocess.run([sys.executable, "-c", code], env=env,
                       capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
