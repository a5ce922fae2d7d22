"""bench.py's command line on the CPU: whatever flags are given, rank 0
prints exactly one JSON line (the GPU leg is replaced by a stub here)."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run(monkeypatch, argv):
    monkeypatch.setattr(bench, "run_csa2", lambda args, world, rank, local: {"metric": bench.METRIC, "value": 1.0})
    monkeypatch.setattr(bench, "run_prefill", lambda args, world, rank, local: {"metric": "prefill", "value": 2.0})
    monkeypatch.setattr(bench, "oracle_baseline", lambda cfg: (4.0, "stub sample"))
    monkeypatch.setattr(sys, "argv", ["bench.py"] + argv)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main()
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1, lines
    return json.loads(lines[0])


def test_one_line_without_the_cpu_baseline(monkeypatch):
    r = _run(monkeypatch, ["--config", "2", "--no-cpu-baseline"])
    assert r["value"] == 1.0 and "cpu_baseline" not in r


def test_one_line_with_the_cpu_baseline(monkeypatch):
    r = _run(monkeypatch, ["--config", "2"])
    assert r["cpu_baseline"]["value"] == 0.25 and r["cpu_baseline"]["kind"] == "oracle"


def test_prefill_line_without_the_cpu_baseline(monkeypatch):
    r = _run(monkeypatch, ["--config", "4", "--no-cpu-baseline"])
    assert r["value"] == 2.0
