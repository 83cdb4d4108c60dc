"""bench.py is single-GPU: asking it for more GPUs is an error before any GPU
work (no GPU needed)."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args,
                          capture_output=True, text=True, env=env, timeout=300)


def test_bench_refuses_more_than_one_gpu():
    r = run_bench(["--gpus", "2", "--steps", "1"])
    assert r.returncode != 0
    assert "one GPU" in r.stderr
