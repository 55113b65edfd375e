"""The benchmark's reference arm (the oracle timed on the host) keeps the JSON
line contract: one line, the decode metric and its unit, a cpu_baseline that
describes the run, an e2e block with no host-device copies. Runs on the CPU
with the tiny workload; the helpers behind the large workloads' bounded
samples (a prompt prefix for prefill, a 1-layer model extrapolated to all
layers for the 8B geometry) run in-process on tiny shapes."""
import json
import os
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


def run_bench(*args, timeout=600):
    env = dict(os.environ)
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    p = subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=timeout)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_line_on_tiny():
    d = run_bench("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3")
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "config"):
        assert k in d, k
    assert d["unit"] == "tok/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_bounded_oracle_samples_on_tiny_shapes():
    sys.path.insert(0, str(ROOT))
    import bench
    from quantized_transformer_decode_gb300 import inputs
    tiny = inputs.WORKLOADS["tiny"]
    assert bench.oracle_prefill_rate(tiny, 16) > 0
    secs, desc = bench.oracle_decode_extrapolated(tiny)
    assert secs > 0 and "extrapolated" in desc
    # the extrapolation of a 1-layer model to 2 layers is of the order of the
    # 2-layer model's own step time
    s2, _ = bench.oracle_decode(tiny, 0, 3, 16)
    assert 0.2 < secs / (s2 / 3) < 5.0


def test_warmup_below_three_is_rejected():
    p = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--warmup", "2"], cwd=ROOT, capture_output=True,
                       text=True, timeout=120)
    assert p.returncode != 0 and "warmup" in p.stderr
