"""bench.py --impl reference on the CPU: the oracle timed as the reference
arm prints the one JSON line the driver reads, and ranks other than 0 of a
replica launch print nothing."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _run(args, rank="0"):
    env = dict(os.environ, RANK=rank, WORLD_SIZE="2" if rank != "0" else "1")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--cpu-seconds",
                           "0.5", "--steps", "3", "--warmup", "3", *args], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=300)


@pytest.mark.parametrize("workload", ["sampling_chain_b32_g8_v32000_bf16", "greedy_chain_b4_g4_v1000_f32",
                                      "tree_kv_compact_b16_n64_d6_w131072"])
def test_reference_line(workload):
    r = _run(["--workload", workload])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert KEYS <= set(line), KEYS - set(line)
    assert line["impl"] == "reference" and line["config"]["workload"] == workload
    assert line["value"] > 0 and line["higher_is_better"] is True and line["vs_baseline"] is None
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # value x ms_per_step is one call's work: draft tokens (B x gamma) or cache rows
    per_call = line["config"].get("rows_per_call") or line["config"]["batch"] * line["config"]["gamma"]
    assert line["value"] * line["ms_per_step"] / 1000.0 == pytest.approx(per_call, rel=1e-9)


def test_other_ranks_print_nothing():
    r = _run(["--workload", "greedy_chain_b4_g4_v1000_f32"], rank="1")
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
