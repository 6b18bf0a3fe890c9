"""The JSON contract of bench.py's reference arm on CPU: the fp64 oracle timed
on the host cores prints one line with impl "reference", the metric, unit and
direction of the fused arm, a cpu_baseline describing the run and an e2e
block with zero host copies.  The oracle's timing itself is replaced by a
fixed result here (the arm's own run takes minutes); what is checked is the
line around it, and that the arm never touches CUDA."""
import argparse
import io
import json
import os
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from coda_inputs import B7  # noqa: E402


def test_reference_arm_line(monkeypatch):
    calls = []

    def fake(shape, target_s=12.0, max_rows=4096):
        calls.append((shape.name, max_rows))
        return {"value": 0.5, "unit": bench.UNIT, "cores": 16, "kind": "oracle",
                "sample": "fp64 numpy oracle block fwd+bwd on 256 rows", "seconds": 1.5, "rows": 256}

    monkeypatch.setattr(bench, "cpu_oracle_baseline", fake)
    monkeypatch.delenv("RANK", raising=False)
    args = argparse.Namespace(gpus=1, steps=2, warmup=3)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, B7)
    lines = [l for l in buf.getvalue().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    assert j["metric"] == bench.METRIC and j["unit"] == bench.UNIT and j["higher_is_better"] is True
    assert j["steps"] == 2 and j["warmup"] == 3 and j["n_gpus"] == 1
    assert j["value"] == 0.5 and j["ms_per_step"] == 1500.0
    assert j["dtype"] == "f64" and j["vs_baseline"] is None
    assert j["config"]["workload"] == B7.name
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 16 and cb["value"] == j["value"] and cb["sample"]
    assert j["e2e"] == {"value": 0.5, "unit": bench.UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert len(calls) == 5  # warm-up and timed steps, each a bounded sample


def test_reference_arm_other_ranks_print_nothing(monkeypatch):
    monkeypatch.setattr(bench, "cpu_oracle_baseline", lambda *a, **k: (_ for _ in ()).throw(AssertionError))
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(argparse.Namespace(gpus=2, steps=2, warmup=3), B7)
    assert buf.getvalue() == ""
