"""The benchmark's reference arm (the CPU oracle timed on a bounded sample)
runs without a GPU: one JSON line with the contract's keys from rank 0, and
nothing from any other rank."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env, *args):
    env = dict(os.environ, **extra_env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_line_with_the_contract_keys():
    r = _run({}, "--workload", "tiny", "--steps", "3", "--warmup", "3", "--ref-sample-tokens", "4")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == "moe_layer_tokens_per_s" and d["unit"] == "tokens/s"
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["tokens"] == 64 and d["config"]["experts"] == 8
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and "first 4" in cb["sample"]
    # the line describes what was timed: K steps of the stated sample
    assert cb["tokens_per_step"] == 4
    assert abs(d["steps"] * d["ms_per_step"] / 1e3 - cb["timed_seconds"]) <= 0.02 + 0.01 * cb["timed_seconds"]
    assert abs(d["value"] - 4 / (d["ms_per_step"] / 1e3)) <= 1e-3 * d["value"] + 1e-3
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--workload", "tiny", "--gpus", "2")
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
