"""The benchmark's oracle arm (`bench.py --impl reference`) on CPU: one JSON
line that keeps the line contract, with exactly the requested warm-up and
timed steps, and a rank other than 0 that exits without work."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", PYTHONDONTWRITEBYTECODE="1",
               **(extra_env or {}))
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                           "--warmup", "1", "--cpu-units", "2"], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_line():
    p = _run()
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and "2 of 288" in d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("8b_128k")


def test_reference_arm_other_ranks_exit_without_work():
    p = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""


def test_extra_workload_failure_keeps_the_line(monkeypatch, capsys):
    """An extra workload that fails (here: the slot-map event, as if the disk
    or the device ran out) is reported under its own key, and the line with
    the headline and the other workloads still prints."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test",
                                                  os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    ran = []

    def ok(name):
        def run(*args, **kw):
            ran.append(name)
            return {"ok": name}
        return run

    def fails(*args, **kw):
        ran.append("slotmap")
        raise OSError("No space left on device")

    monkeypatch.setattr(bench, "run_ours", lambda *a: {"metric": "m", "value": 1.0})
    monkeypatch.setattr(bench, "peaks", lambda: (6702.8, 1910.5))
    monkeypatch.setattr(bench, "config_event", lambda args, dev, name, peak: ok(name)())
    monkeypatch.setattr(bench, "slot_map_event", fails)
    for fn, name in (("tiered_event", "tiered"), ("repo_event", "repo"),
                     ("paged_event", "paged"), ("confidence_monitor", "confidence")):
        monkeypatch.setattr(bench, fn, ok(name))
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    bench.main()
    out = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(out) == 1
    d = json.loads(out[0])
    assert ran == ["27b_1m", "ragged_128", "slotmap", "tiered", "repo", "paged", "confidence"]
    assert d["value"] == 1.0 and d["slotmap_event"] == {"error": "OSError: No space left on device"}
    assert d["event_27b_1m"] == {"ok": "27b_1m"} and d["confidence_monitor"] == {"ok": "confidence"}
