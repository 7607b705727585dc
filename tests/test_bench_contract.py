"""The benchmark's command-line contract on CPU: defaults, and the reference
arm's JSON line (the CPU oracle on a bounded sample), which needs no GPU."""

import io
import json
import sys
from contextlib import redirect_stdout

import bench


def test_defaults(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse_args()
    assert a.gpus == 1 and a.impl == "ours" and a.warmup >= 3 and a.steps >= 1


def test_reference_line(monkeypatch):
    for v in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "2", "--warmup", "0"])
    args = bench.parse_args()
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    lines = [x for x in buf.getvalue().splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "steps/s"
    assert d["value"] > 0 and d["steps"] == 2 and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["config"]["workload"] == bench.DEFAULT_WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_step_bytes_count_rows_read_and_written():
    m, n, H, V = 3072, 60, 4096, 128256
    # rows read + packed written, logits, hiddens, one verify row, bitmap read and written, I_t
    assert bench.step_bytes(m, n, H, V) == 2 * m * H * 2 + n * m * 4 + n * H * 2 + V * 4 + 2 * 16032 + 4 * m
    assert bench.proj_bytes(m, n, H) == bench.step_bytes(m, n, H, V) - V * 4 - 2 * 16032


def test_single_thread_oracle_sample():
    d = bench.single_thread_oracle(bench.DEFAULT_WORKLOAD, steps=2)
    assert d is not None and d["cores"] == 1 and d["value"] > 0 and d["unit"] == "steps/s"
