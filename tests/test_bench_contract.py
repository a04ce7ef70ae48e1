"""bench.py's reference arm (the fp64 oracle on the host cores) prints one contract line."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line_on_the_tiny_workload():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                          "--steps", "2", "--warmup", "3"], cwd=ROOT, capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["n_gpus"] == 1 and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "tiny_w2_c512"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_fewer_than_three_warmup_steps_refused():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                          "--steps", "1", "--warmup", "2"], cwd=ROOT, capture_output=True,
                         text=True, timeout=300)
    assert out.returncode != 0 and "warmup" in out.stderr
