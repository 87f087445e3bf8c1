"""bench.py's CPU side: the oracle sample it times for the CPU baseline and the
JSON line of its reference arm (the oracle on host cores).  No GPU."""
import io
import json
import types
from contextlib import redirect_stdout

import bench
import ragen


def test_cpu_oracle_sample_times_real_rows():
    wl = ragen.WORKLOADS["noncausal_8k"]
    r = bench.cpu_oracle_sample(wl, 0.5)
    assert r["rows"] > 0 and r["seconds"] > 0 and r["threads"] >= 1
    # every sampled row of the non-causal workload sees all S keys
    assert r["flops"] == 4.0 * wl.D * wl.S * r["rows"]


def test_reference_arm_prints_one_contract_line(monkeypatch):
    wl = ragen.WORKLOADS["gqa_128k"]
    # a stub sample keeps this test fast; its figures pass straight through
    monkeypatch.setattr(bench, "cpu_oracle_sample",
                        lambda wl_, s: {"flops": 2e12, "seconds": 4.0, "rows": 64, "threads": 8})
    args = types.SimpleNamespace(gpus=1, steps=2, warmup=1, workload="gqa_128k")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.reference_arm(args, wl) == 0
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] == 2 * 2e12 / (2 * 4.0) / 1e12  # two timed steps of the stub
    assert d["ms_per_step"] == 4000.0
    assert d["config"]["workload"] == wl.name
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 8 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
