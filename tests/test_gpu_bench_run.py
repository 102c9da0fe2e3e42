"""`bench.py` end to end at a reduced batch (16 requests): every leg runs and the JSON line keeps
the contract's keys. Reduced batches are how profiling runs call the bench; the KV-commit leg
once failed there because it borrowed the verify legs' handle, sized for 16 requests."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_reduced_batch_runs_every_leg():
    r = subprocess.run([sys.executable, "bench.py", "--steps", "3", "--warmup", "3", "--requests",
                        "16", "--skip-e2e", "--skip-cpu-baseline", "--skip-parity"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "dtype", "config", "roofline", "gpu_launches",
              "clocks"):
        assert k in line, k
    assert line["config"]["global_batch"] == 16
    assert line["value"] > 0 and line["gpu_launches"] > 0
    # the DRAM record covers the full batch only
    assert line["roofline"]["traffic"] is None and "traffic_note" in line["roofline"]
    for leg in ("kv_commit", "dense_chain", "small_tries", "high_accept", "adaptive_budget"):
        assert leg in line and line[leg], leg
    for cache in ("bf16", "fp8_e4m3", "fp8_e4m3_scale_0.0173"):
        assert line["kv_commit"][cache]["ms_per_call"] > 0
