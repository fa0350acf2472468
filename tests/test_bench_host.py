"""bench.py's host-side contract without a GPU: the reference arm (the
oracle timed on the host cores) prints one JSON line with the same metric,
unit, direction and workload config as the GPU arm, plus its cpu_baseline
and an end-to-end entry with no device copies.  The oracle sample itself is
replaced by a stub here so the test takes no time."""
import contextlib
import io
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class _Args:
    steps, warmup, gpus = 3, 3, 1


def test_reference_arm_line(monkeypatch):
    calls = []

    def stub(seconds=12.0):
        calls.append(seconds)
        return 0.025, 16, "stub sample", 0.01

    monkeypatch.setattr(bench, "oracle_sample", stub)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(_Args, 0, 1)
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"] == bench.step_config()
    assert d["steps"] == 3 and d["warmup"] == 3 and len(calls) == 6
    assert d["value"] == 0.025
    assert d["cpu_baseline"] == {"value": 0.025, "unit": "TFLOP/s", "cores": 16, "kind": "oracle",
                                 "sample": "stub sample"}
    assert d["e2e"] == {"value": 0.025, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_step_config_counts_the_algorithmic_work():
    c = bench.step_config()
    # scale-up prefill: 36 caches x 32 heads x 4 d FLOP per visible pair
    assert abs(c["prefill_gflop_per_step"] - 6842.33588736) < 1e-6
    # batch-64 verify: K/V of every visible key per (cache, kv head), Q, O and the block
    assert abs(c["verify_mb_per_step"] - 842.79296) < 1e-6
    # insert: the new frames read and written, K and V, 36 caches
    assert abs(c["insert_mb_per_step"] - 452.984832) < 1e-6
