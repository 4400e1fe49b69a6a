"""The N > 1 path of bench.py (independent replicas, no data-path collective):
its host-side pieces run as two gloo ranks on the CPU -- the barrier, the
max-over-ranks timing, and the reference arm printing on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
world, rank, local = bench.dist_setup(None)
assert world == 2
bench.barrier(world)
t = bench.max_over_ranks(world, 1.0 + rank)          # rank 1 is the slower one
print(json.dumps({{"rank": rank, "max": t}}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def _spawn(code, extra_env=None, nproc=2):
    port = _free_port()
    procs = []
    for r in range(nproc):
        env = dict(os.environ, WORLD_SIZE=str(nproc), RANK=str(r), LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=240)
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_barrier_and_max_over_ranks():
    outs = _spawn(WORKER.format(root=ROOT))
    vals = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(v["rank"] for v in vals) == [0, 1]
    assert all(v["max"] == 2.0 for v in vals)          # every rank sees the slowest time


REFERENCE = r"""
import sys
sys.path.insert(0, {root!r})
sys.argv = ["bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0",
            "--gpus", "2"]
import bench
bench.main()
"""


def test_reference_arm_prints_on_rank_zero_only():
    outs = _spawn(REFERENCE.format(root=ROOT))
    lines = [[l for l in o.splitlines() if l.startswith("{")] for o in outs]
    assert len(lines[0]) == 1 and lines[1] == []
    rec = json.loads(lines[0][0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
