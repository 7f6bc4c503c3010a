"""Host-side logic of bench.py's CPU leg (no GPU): the oracle worker pool and its arithmetic.

The pool times the oracle's decode in spawned worker processes, one (layer, sequence, kv-head)
unit each, all at once; their token rates add.  Units timed one after another in one thread give
total tokens over total time instead.
"""

import numpy as np
import pytest

import bench
from kv_cache_quantization_append_gb300 import synth


def test_rates_add_only_for_concurrent_workers():
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    layers, lens = w["n_layers"], np.array([32768])
    step_token_heads = 32768 * w["n_kv_heads"] * layers
    res = [(1000, 1.0, 3), (3000, 2.0, 5)]                 # (tokens, seconds, calls) per unit
    conc = bench._baseline_record(w, layers, lens, res, 2, 1.0, True)
    assert conc["cores"] == 2
    assert conc["value"] == pytest.approx(32768 / (step_token_heads / 2500.0))
    assert conc["per_core_value"] == pytest.approx(32768 / (step_token_heads / 1250.0))
    seq = bench._baseline_record(w, layers, lens, res, 1, 1.0, False)
    assert seq["cores"] == 1
    assert seq["value"] == pytest.approx(32768 / (step_token_heads / (4000 / 3.0)))
    assert seq["value"] == seq["per_core_value"]


def test_step_covers_the_timed_layers_only():
    """The ragged 27B-shaped workload times one allocated layer: the baseline scales to that layer."""
    w, layers, lens = bench.workload_cfg("dense27b-ragged-b32")
    assert layers == 1 < w["n_layers"]
    rec = bench._baseline_record(w, layers, lens, [(1000, 1.0, 1)], 1, 1.0, False)
    assert rec["value"] == pytest.approx(1000 / w["n_kv_heads"])
    assert f"of the {len(lens) * w['n_kv_heads']} in one step" in rec["sample"]


def test_host_cores_is_capped():
    n = bench.host_cores()
    assert 1 <= n <= bench.ORACLE_MAX_WORKERS


def test_oracle_worker_pool_on_the_tiny_workload():
    w, layers, lens = bench.workload_cfg("tiny")
    timer = bench.OracleTimer(w, layers, lens, 2)
    try:
        res = timer.step(0.2)
        assert len(res) == 2
        for tokens, secs, calls in res:
            assert calls >= 1 and tokens == calls * int(lens[0]) and secs > 0
        cb = bench.cpu_baseline(w, layers, lens, timer=timer, budget_s=0.2)
        assert cb["cores"] == 2 and cb["kind"] == "oracle" and cb["value"] > 0
        assert "2 spawned processes" in cb["sample"]
    finally:
        timer.close()
    assert all(not p.is_alive() for p in timer.workers)


def test_one_thread_fallback():
    w, layers, lens = bench.workload_cfg("tiny")
    cb = bench.cpu_baseline(w, layers, lens, budget_s=0.3, pool=False)
    assert cb["cores"] == 1 and cb["value"] > 0 and "one thread" in cb["sample"]


def test_reference_arm_json_line(monkeypatch):
    """--impl reference: rank 0 prints the contract's line, timed on the oracle; other ranks none."""
    import argparse

    monkeypatch.setattr(bench, "REFERENCE_WALL_S", 1.0)
    monkeypatch.setattr(bench, "host_cores", lambda: 2)
    args = argparse.Namespace(steps=1, warmup=3, workload="tiny", impl="reference", gpus=1)
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(args) is None
    monkeypatch.setenv("RANK", "0")
    res = bench.run_reference(args)
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in res, key
    assert res["impl"] == "reference" and res["steps"] == 1 and res["warmup"] == 3
    assert res["value"] > 0 and res["higher_is_better"] is True and res["vs_baseline"] is None
    assert res["config"]["workload"] == "tiny"
    cb = res["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["value"] == res["value"] and cb["sample"]
    e2e = res["e2e"]
    assert e2e["value"] == res["value"] and e2e["unit"] == res["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert res["ms_per_step"] == pytest.approx(512 / res["value"] * 1e3)
