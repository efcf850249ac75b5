"""Host-side pieces of the benchmark that need no GPU."""

import pytest

import bench


@pytest.mark.parametrize("layers", [1, 2, 5, 21, 32, 100])
def test_copy_runs_cover_the_layers_in_order(layers):
    runs = bench.copy_runs(layers)
    assert runs[0] == (0, 1)
    assert runs[-1][1] == layers
    for (a, b), (c, _) in zip(runs, runs[1:]):
        assert b == c and a < b
    # each full run is four times the one before it
    sizes = [b - a for a, b in runs]
    for s0, s1 in zip(sizes[:-2], sizes[1:-1]):
        assert s1 == 4 * s0


def test_copy_runs_of_the_llama_step():
    assert bench.copy_runs(32) == [(0, 1), (1, 5), (5, 21), (21, 32)]


def test_reference_arm_prints_one_contract_line():
    # the reference arm times the CPU oracle; it needs no GPU
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=root, check=True).stdout
    lines = [l for l in out.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == bench.WORKLOADS["llama8b_eagle"]
    # whole steps are timed: the line's time is what the steps took
    assert d["steps"] == 1 and "whole oracle steps" in d["cpu_baseline"]["sample"]


def test_both_arms_print_the_same_config():
    import bench
    from synth import make_case
    for name in ("llama8b_eagle", "tiny"):
        case, _ = bench.build_case(name, with_logits=False)
        cfg = bench.workload_config(name, case)
        assert cfg["workload"] == bench.WORKLOADS[name]
        assert set(cfg) == {"workload", "layers", "batch", "total_nodes", "seed", "l2", "parallelism"}
