"""bench.py's reference arm (the fp64 oracle timed on the host cores) keeps the
one-line JSON contract, alone and as two ranks, where rank 0 alone prints."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CMD = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
       "--warmup", "0"]


def check_line(d, n_gpus):
    assert d["impl"] == "reference"
    assert d["metric"] == "attended keys/s (GQA decode over int4 KV cache)"
    assert d["unit"] == "keys/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == n_gpus and d["steps"] == 1 and d["warmup"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_reference_arm_one_process():
    env = dict(os.environ)
    for key in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(key, None)
    out = subprocess.run(CMD, env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    check_line(json.loads(lines[0]), 1)


def test_reference_arm_two_ranks_rank0_prints():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                   RANK=str(rank), LOCAL_RANK=str(rank))
        procs.append(subprocess.Popen(CMD + ["--gpus", "2"], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=600)
        assert p.returncode == 0, err[-2000:]
        outs.append([l for l in out.splitlines() if l.startswith("{")])
    assert len(outs[0]) == 1 and outs[1] == []
    check_line(json.loads(outs[0][0]), 2)
