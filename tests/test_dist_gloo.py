"""The multi-process path of the benchmark, on CPU with the gloo backend and two
ranks: the rank helpers behind the barrier, max-over-ranks timing and the
whole-job sum, and the reference arm's rule that rank 0 alone runs and prints
under torchrun.  (The GPU path shards nothing: every rank is an independent
replica, so these host-side pieces are all that N > 1 adds.)"""
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


_RANK_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import bench
d = bench.Dist()
d.init(use_gpu=False)
r = d.rank
d.barrier()
out = {"rank": r, "world": d.world, "max": d.max(1.5 + r), "sum": d.sum(10.0 * (r + 1))}
d.close()
print(json.dumps(out))
"""


def test_rank_helpers_two_gloo_ranks():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_SCRIPT, ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        so, se = p.communicate(timeout=180)
        assert p.returncode == 0, se[-2000:]
        outs.append(json.loads(so.strip().splitlines()[-1]))
    for o in outs:
        assert o["world"] == 2
        assert o["max"] == 2.5   # the slowest rank's time
        assert o["sum"] == 30.0  # the whole job's units
    assert sorted(o["rank"] for o in outs) == [0, 1]


def test_reference_arm_rank0_alone_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "quantize",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--reference-seconds", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1  # rank 0 only
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
