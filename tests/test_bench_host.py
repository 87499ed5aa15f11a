"""The benchmark's CPU-baseline leg on a small workload (CPU only): the
reported keys, units and sample description, the one-thread figure, and
that the oracle's thread count is restored afterwards."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from speculative_decoding_verify_causal_gb300 import workloads as wl  # noqa: E402


def test_cpu_baseline_line_on_the_small_workload():
    w = wl.config_workload("tiny")
    cores = oracle.max_threads(0)
    cb = bench.cpu_baseline(w, wl, min_seconds=0.3)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s"
    assert cb["value"] > 0 and cb["seconds"] >= 0.3
    assert cb["cores"] == cores
    assert "query rows" in cb["sample"] and "fp64" in cb["sample"]
    st = cb["single_thread"]
    assert st["unit"] == "GB/s" and st["value"] > 0
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    # the one-thread run must not leave the oracle on one thread
    assert oracle.max_threads(0) == cores


def test_cpu_model_is_a_nonempty_string():
    m = bench.cpu_model()
    assert isinstance(m, str) and len(m) > 0


def test_reference_arm_prints_one_contract_line():
    # `bench.py --impl reference` times the fp64 oracle on the host cores and
    # prints one JSON line with the reference-arm keys (CPU only)
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("tiny")


def test_default_run_keeps_the_warmup_rule():
    # the driver's default invocation: at least 3 untimed warm-up steps
    old = sys.argv
    try:
        sys.argv = ["bench.py"]
        a = bench.parse_args()
    finally:
        sys.argv = old
    assert a.warmup >= 3 and a.steps >= 1 and a.gpus == 1 and a.impl == "ours" and a.config == "lookup16"
