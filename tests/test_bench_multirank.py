"""bench.py's N>1 path on CPU: two gloo ranks under torchrun (127.0.0.1)."""
import json
import os
import socket
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout=300):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=%d" % _free_port()] + args
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def test_max_over_ranks_and_whole_job_value():
    lines = _torchrun([os.path.join(HERE, "multirank_probe.py")])
    assert sorted(l["rank"] for l in lines) == [0, 1]
    for l in lines:
        assert l["world"] == 2
        assert l["max"] == [2.0, 20.0, 0.5]          # elementwise max over the two ranks
        assert l["value"] == 8192 * 2 / 2.0          # all ranks' units / slowest time


def test_reference_arm_prints_once_under_torchrun():
    lines = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                       "--warmup", "0"])
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
