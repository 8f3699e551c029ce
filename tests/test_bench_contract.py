"""The benchmark's JSON line on the CPU: the reference arm (the oracle on the
host cores) runs without a GPU, so its line is checked here against the keys
the contract asks for; the CUDA arm's config helper is checked directly."""
import json
import os
import subprocess
import sys
from types import SimpleNamespace

from tests.conftest import ROOT


def test_reference_arm_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
           "--warmup", "0", "--cpu-sample-seconds", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["higher_is_better"] is True and d["value"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["config"]["workload"].startswith("decode: 48 QMoE layers H=2048 inter=768 E=128 k=8 INT4 b32")
    assert d["config"]["passes"] == 12
    # the prefill half of the metric: the oracle on a sample of the 8K prefill tokens
    pf = d["prefill"]
    assert pf["value"] > 0 and pf["cpu_baseline"]["kind"] == "oracle" and "prefill tokens" in pf["cpu_baseline"]["sample"]


def test_reference_arm_rejects_options():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--options"]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert r.returncode != 0 and "CUDA arm only" in r.stderr


def test_workload_config_names_options():
    import bench
    import synthetic

    shape, _, _ = synthetic.decode_layer(8)
    base = bench.workload_config(SimpleNamespace(workload="decode", options=False, passes=12), shape, 48, 1)
    opt = bench.workload_config(SimpleNamespace(workload="decode", options=True, passes=12), shape, 48, 1)
    assert "options" not in base and "biases" in opt["options"]
    assert base["parallelism"] == "replicas x1" and base["T"] == 8 and base["layers"] == 48
    assert base["passes"] == 12 and "12 passes" in base["step"]
    one = bench.workload_config(SimpleNamespace(workload="prefill", options=False, passes=12), shape, 1, 1)
    assert one["passes"] == 1
