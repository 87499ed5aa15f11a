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
