"""`bench.py --impl reference` (the CPU oracle timed on every host core) on
CPU: its one JSON line keeps the benchmark's keys and the headline workload's
config, warm-up and timed steps are the ones asked for, a slow host gets a
smaller row sample per step instead of a longer run, and ranks other than 0 do
no work."""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "rows/s" and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 3          # at least three warm-up steps
    assert line["value"] > 0 and line["n_gpus"] == 1 and line["scaling"] == "weak"
    assert line["config"]["global_batch"] == 16384 and line["config"]["seq_len"] == "28673..32768"
    assert line["config"]["workload"].startswith("RAGGED prefill extend")
    base = line["cpu_baseline"]
    import oracle
    assert base["kind"] == "oracle" and base["cores"] == oracle.host_cores() and base["value"] == line["value"]
    assert "2 timed step(s) after 3 warm-up step(s)" in base["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def _bench():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    return bench


def test_reference_arm_samples_rows_on_a_slow_host(capsys, monkeypatch):
    bench = _bench()
    monkeypatch.setattr(bench, "REF_BUDGET_S", 1e-3)
    bench.run_reference(argparse.Namespace(steps=2, warmup=3, gpus=1), None, 0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert "the oracle over 1 of rows 2048..2303" in line["cpu_baseline"]["sample"]
    assert line["value"] > 0


def test_reference_arm_other_ranks_do_nothing(capsys):
    bench = _bench()
    bench.run_reference(argparse.Namespace(steps=2, warmup=3, gpus=2), None, 1)
    assert capsys.readouterr().out == ""
