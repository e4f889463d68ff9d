"""The multi-rank bench path on CPU (world size 2, gloo; no GPU).

Every rank runs an independent replica of the decode step; the process group carries
only the barriers around the timed region and the max of the ranks' step times, and the
reported value is the units all ranks processed over that max.  These tests run the
bench's own helpers in two processes over gloo on 127.0.0.1.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys, time
sys.path.insert(0, os.environ["ROOT"])
import bench
rank, world, local, pg = bench.dist_init(None, backend="gloo")
assert (rank, world) == (int(os.environ["RANK"]), 2), (rank, world)
# a slower rank: its time must become everyone's
dt_local = 0.010 * (1 + rank)
bench.barrier(pg)
dt = bench.max_over_ranks(pg, dt_local)
bench.barrier(pg)
print(json.dumps({"rank": rank, "dt": dt, "value": world * 1.0 / dt}), flush=True)
pg.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank: int, world: int, port: int) -> dict:
    env = dict(os.environ)
    env.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), ROOT=ROOT,
               CUDA_VISIBLE_DEVICES="")
    return env


def test_two_rank_barrier_and_max_over_ranks():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", WORKER], env=_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["dt"] == 0.020  # the slower rank's time, on both ranks
        assert o["value"] == 2 / 0.020  # whole-job: both ranks' tokens over the max time


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun the oracle is timed on rank 0 alone; rank 1 prints nothing and exits
    0 without touching a process group (no peer is waiting for it)."""
    for workload in ("step", "slots"):
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--workload", workload, "--steps", "1", "--warmup", "3"],
                           env=_env(1, 2, _free_port()), capture_output=True, text=True, timeout=120)
        assert r.returncode == 0, r.stderr[-2000:]
        assert r.stdout.strip() == ""


def test_single_rank_needs_no_process_group():
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "-c",
                        "import sys; sys.path.insert(0, %r); import bench; "
                        "rk, w, l, pg = bench.dist_init(None, backend='gloo'); "
                        "assert (rk, w, l, pg) == (0, 1, 0, None); "
                        "assert bench.max_over_ranks(pg, 0.5) == 0.5; bench.barrier(pg)" % ROOT],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
