"""The benchmark's JSON line, checked on CPU through its reference arm (the
fp64 oracle timed on the host cores): one line, with the keys and types the
line's readers expect."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_prints_one_contract_line():
    d = _run("--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3", "--ref-budget", "2")
    assert d["impl"] == "reference"
    for k, t in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                 ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                 ("dtype", str), ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)):
        assert isinstance(d[k], t), (k, d[k])
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["scaling"] == "weak" and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "tiny-fp32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_too_few_warmup_steps_are_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_workload_overrides_reach_the_line():
    """--batch / --layers (smaller or larger cases of a workload, for
    profiling) change the measured configuration, and the line says so."""
    d = _run("--impl", "reference", "--config", "1", "--batch", "2", "--layers", "2", "--steps", "2",
             "--warmup", "3", "--ref-budget", "2")
    assert d["config"]["workload"] == "tiny-fp32"
    assert d["config"]["batch"] == 2
    one = _run("--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3", "--ref-budget", "2")
    assert one["config"]["batch"] == 1
    assert d["config"]["stitched_tokens_per_step"] > one["config"]["stitched_tokens_per_step"]
