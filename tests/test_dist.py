"""Multi-process path of bench.py on CPU: world size 2 over gloo.

The step shards by request with no exchange on the data path, so the only cross-rank
operations are the timing barrier and the max over ranks; these tests run them as two
gloo ranks on host cores, and launch bench.py under torch.distributed.run the way a
multi-GPU run does (rank 0 alone prints the JSON line).
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


RANK_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, os.environ["PKV_ROOT"])
import bench
d = bench.Dist()
assert d.world == 2 and d.pg is not None
d.barrier()
# every rank reports its own time; all must see the slowest
m = d.max(1.5 + d.rank)
d.barrier()
print(json.dumps({"rank": d.rank, "max": m}))
d.close()
"""


def _env(rank, port):
    e = dict(os.environ)
    e.update(PKV_ROOT=ROOT, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
             MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    return e


def test_dist_max_over_ranks_gloo():
    port = free_port()
    procs = [subprocess.Popen([sys.executable, "-c", RANK_SCRIPT], env=_env(r, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, e
        outs.append(json.loads(o.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["max"] == 2.5 for o in outs)


def test_bench_reference_arm_two_ranks():
    """torchrun, 2 ranks: rank 0 prints exactly one JSON line, rank 1 does no work, both
    exit 0."""
    port = free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3"]
    r = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2 and line["steps"] == 1 and line["warmup"] == 3
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
