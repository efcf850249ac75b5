"""The benchmark is single-GPU: a multi-GPU launch of the GPU arm is refused
before the library is loaded (its paired attention kernel shares K/V tiles
between the CTAs of a cluster with TMA multicast, kept to one-GPU jobs); the
reference arm (CPU only) prints from rank 0 and the other ranks exit quietly."""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("argv,env", [
    (["--gpus", "2"], {}),
    (["--gpus", "8"], {}),
    ([], {"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"}),
    ([], {"WORLD_SIZE": "4", "RANK": "3", "LOCAL_RANK": "3"}),
])
def test_multi_gpu_launch_is_refused_before_loading_the_library(argv, env):
    e = dict(os.environ, **env)
    # a marker module on the path records whether torch got imported
    r = subprocess.run([sys.executable, "-c",
                        "import sys, bench\n"
                        "try:\n"
                        "    bench.main(sys.argv[1:])\n"
                        "except SystemExit as ex:\n"
                        "    print('torch' in sys.modules, 'speculative_decoding_tree_sv_gb300.binding' in sys.modules)\n"
                        "    raise\n"] + argv + ["--steps", "1"],
                       capture_output=True, text=True, timeout=120, cwd=ROOT, env=e)
    assert r.returncode == 2
    assert "one GPU only" in r.stderr
    assert r.stdout.strip() == "False False"


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    import argparse

    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(config="tiny", steps=1, warmup=3, gpus=2, reference_budget_s=10.0)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_reference_plan_times_whole_steps_within_the_budget():
    import bench
    assert bench.reference_plan(20, 5, 2.2, 200.0) == 20
    assert bench.reference_plan(1000, 10, 2.2, 200.0) == 90
    assert bench.reference_plan(5, 3, 500.0, 200.0) == 1  # at least one


def test_clock_summary_skips_idle_samples():
    import bench
    lines = ["2070, 2070, 500, 0x0, Not Active, Not Active, Not Active, Not Active, Not Active",
             "345, 2070, 100, 0x1, Not Active, Not Active, Not Active, Not Active, Active",
             "1965, 2070, 900, 0x4, Not Active, Not Active, Not Active, Active, Not Active",
             "garbage"]
    s = bench.summarize_clocks(lines)
    assert s["sm_mhz"] == (2070 + 1965) / 2 and s["samples"] == 2 and s["samples_total"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.summarize_clocks([])["reasons"] == ["unsampled"]
