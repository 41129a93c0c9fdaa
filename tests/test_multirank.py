"""The replica path of bench.py on two CPU ranks (gloo): process-group setup
from the torchrun environment, the barriers around the timed region and the
max-over-ranks reduction of the per-rank times, as a two-GPU run uses them.
The decode path has no exchange between (sequence, KV head) units, so ranks
are replicas and these are the only collectives."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["KVQ_ROOT"])
import bench
world, rank, local = bench.dist_setup()
bench.barrier(world)
slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)   # rank 1 is the slower one
bench.barrier(world)
import torch.distributed as dist
dist.destroy_process_group()
print(json.dumps({"world": world, "rank": rank, "local": local, "slowest": slowest}))
"""


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_rank_barrier_and_max_over_ranks():
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                   RANK=str(rank), LOCAL_RANK=str(rank), KVQ_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    results = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        results.append(json.loads(out.strip().splitlines()[-1]))
    results.sort(key=lambda r: r["rank"])
    assert [r["rank"] for r in results] == [0, 1]
    assert all(r["world"] == 2 for r in results)
    assert [r["local"] for r in results] == [0, 1]
    # every rank reports the slowest rank's time
    assert all(r["slowest"] == 15.0 for r in results)


def test_single_process_needs_no_process_group():
    env = dict(os.environ, KVQ_ROOT=ROOT)
    for key in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(key, None)
    out = subprocess.run([sys.executable, "-c", WORKER.replace(
        "import torch.distributed as dist\ndist.destroy_process_group()\n", "")],
        env=env, capture_output=True, text=True, timeout=180)
    assert out.returncode == 0, out.stderr[-2000:]
    r = json.loads(out.stdout.strip().splitlines()[-1])
    assert r == {"world": 1, "rank": 0, "local": 0, "slowest": 10.0}
