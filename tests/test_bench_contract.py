"""bench.py's reference arm on the CPU: the oracle timed on the host's cores prints one JSON line
with every key the line format requires (the GPU arm's line is checked on the GPU machine by running
it); a run with fewer than 3 warm-up steps is refused."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_line():
    r = run_bench("--impl", "reference", "--steps", "3", "--warmup", "3", "--ref-elements", "4000000",
                  "--ref-ns-size", "512")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["ms_per_step"] > 0 and d["ns"]["value"] > 0  # K timed steps of the sample, averaged
    assert isinstance(d["config"]["workload"], str) and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == os.cpu_count() and cb["value"] == d["value"] and cb["sample"]
    assert cb["cpu_model"] and d["adamw_part"]["elements"] == 4_000_000
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_too_few_warmup_steps_refused():
    r = run_bench("--impl", "reference", "--steps", "3", "--warmup", "2", timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr
