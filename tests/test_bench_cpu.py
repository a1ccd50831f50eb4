"""bench.py's launch contract on the CPU: `--gpus N` without a torchrun
environment starts N ranks itself (one engine per GPU in the real run; here
the CPU reference arm, where rank 0 alone measures and prints the line)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gpus_n_spawns_n_ranks():
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--shape", "tiny", "--B", "4", "--steps", "2", "--warmup", "1", "--ctx-lo", "16",
                        "--ctx-hi", "64"], capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "bench rank 0 of 2" in r.stderr and "bench rank 1 of 2" in r.stderr, r.stderr[-2000:]
    lines = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    ln = lines[0]
    assert ln["impl"] == "reference" and ln["n_gpus"] == 2 and ln["steps"] == 2
    assert ln["value"] > 0 and ln["cpu_baseline"]["kind"] == "oracle"
