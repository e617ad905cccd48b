"""The benchmark's host logic on CPU: workload table, the bounded oracle arm,
and the rule that a profiled DRAM traffic figure is used only for the source
it was taken on."""
import json
import os
import subprocess
import sys

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_workloads_name_existing_configs():
    b = _bench()
    assert b.DEFAULT_WORKLOAD in b.WORKLOADS
    for name, (key, metric, workload, keep) in b.WORKLOADS.items():
        assert key in synth.CONFIGS, name
        assert metric and workload, name
        assert keep is None or 0.0 < keep < 1.0, name


@pytest.mark.parametrize("workload", ["vitb16-64f384", "vitl16-16f256-masked50"])
def test_reference_arm_declines_unbounded_or_masked_workloads(workload):
    """Above the token bound (or for the masked workload) the oracle arm prints
    one 'unavailable' line and exits 0 without running the oracle."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload, "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "unavailable" in line


def test_traffic_used_only_for_the_profiled_source():
    b = _bench()
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["attention"]
    got = b._traffic_for("attention", rec["launch"])
    if rec["source_sha"] == b._source_sha(rec["sources"]):
        assert got == rec["dram_bytes_per_launch"]
    else:
        assert got is None
    assert b._traffic_for("attention", "another launch") is None
    assert b._traffic_for("no such kernel", rec["launch"]) is None
