"""bench.py without a GPU: the reference arm (the fp64 oracle timed on the
host cores) prints one JSON line with the keys the benchmark contract asks
for, and the unmasked-FLOP count matches the long-context figures
(14 D per kept pair, S(S+1)/2 kept pairs per head)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_unmasked_flop_count():
    B, H, S, D = 1, 32, 262144, 128
    assert abs(bench._flops(B, H, S, D, 4) - 5.630e14) / 5.630e14 < 1e-3
    assert abs(bench._flops(B, H, S, D, 14) - 1.970e15) / 1.970e15 < 1e-3
    assert bench._flops(1, 1, 1, 1, 14) == 14  # one token keeps one pair
    # whole-job throughput of independent replicas: world x per-rank work / slowest time
    assert bench.job_tflops(2e12, 1000.0, 2) == 4.0


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "1", "--cpu-sample", "512"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"]
    assert line["config"]["S"] == 262144 and line["config"]["N"] == 8
