"""bench.py's reference arm (the oracle timed on host cores) and its JSON
contract, run on the CPU: one line with the same metric and config as the
GPU arm, a cpu_baseline describing the run, an e2e object with no copies,
and no output from ranks other than 0."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.strip()]


def test_reference_arm_json_line():
    lines = _run()
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"] == bench.workload_desc()
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    assert _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


def test_profile_counters_only_for_the_source_they_were_taken_on(monkeypatch):
    # roofline.traffic and the issue view come from the committed ncu figures only while the kernel source
    # hash matches the one they were taken on
    import bench
    prof = {(k, M): bench.measured_profile(f"axis1_k{k}_M{M}") for k in bench.KS for M in bench.MS}
    if not all(prof.values()):  # the source changed since the capture: the bench reports traffic null
        pytest.skip("profiles/traffic.json was taken on other axis-1 kernel sources")
    for (k, M), d in prof.items():
        algorithmic = bench.R * bench.C * k / 8 + 2 * bench.R + 2 * M * bench.C + 2 * M * bench.R
        assert 0.99 <= d["dram_bytes_per_launch"] / algorithmic <= 1.01, "DRAM traffic equals algorithmic bytes"
        assert d["warp_instructions_per_launch"] > 0
    monkeypatch.setattr(bench, "kernel_source_hash", lambda *names: "0" * 16)
    assert bench.measured_profile("axis1_k2_M1") is None
