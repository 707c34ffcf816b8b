"""Host-side checks of bench.py's output contract (no GPU).

The bench prints exactly one JSON line on stdout, and whatever reads it may
keep only the tail of the output, so that line must stay small (the detail
goes to a file). The timed region must hold exactly --steps steps after
exactly --warmup warm-up steps, built from graphs of whole steps.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

MAX_LINE = 2048


def _fake_headline(**over):
    args = dict(
        value=5.9e10, ms_per_step=0.0089, steps=20, warmup=5, n_gpus=1,
        config={"workload": "all7_4096x128", "num_envs": 4096, "seq_len": 128,
                "estimators": 7, "bytes_per_step": 60817408,
                "l2": "inputs larger than L2: 8 rotating buffer sets, 487 MB = 3.8x L2",
                "launch": "seven rlcs_* calls per step on seven streams (fork/join per "
                          "graph); CUDA graphs of whole steps",
                "parallelism": "weak: each rank its own batch"},
        step_gbs=6830.0, peak=6789.3,
        roofline={"bound": "hbm", "achieved": 3980.0, "peak": 6789.3, "unit": "GB/s",
                  "frac": 0.586, "traffic": 10512640, "kernel": "retrace",
                  "bytes_per_launch": 12599296, "us_per_launch": 3.17,
                  "peak_source": "measured hbm_gbs (copy burst)"},
        cpu={"value": 1.2e8, "unit": "env-steps/s", "cores": 16, "kind": "oracle",
             "sample": "123 full 4096x128 batches, all seven estimators, float64 C oracle, "
                       "rows split over 16 threads, 10.0 s",
             "single_thread": {"value": 4.9e7}},
        e2e={"value": 4.8e9, "unit": "env-steps/s", "h2d_bytes_per_step": 14700000,
             "d2h_bytes_per_step": 16800000, "ms_per_step": 0.11, "path": "x" * 500},
        launches=140, clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [],
                              "samples": 12},
        detail_path="bench_detail.json")
    args.update(over)
    return bench.headline_line(**args)


def test_headline_is_one_small_json_line_with_the_contract_keys():
    line = _fake_headline()
    assert "\n" not in line and len(line) <= MAX_LINE, len(line)
    d = json.loads(line)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in d["roofline"], key
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in d["cpu_baseline"], key
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in d["e2e"], key
    assert d["config"]["workload"] == "all7_4096x128"
    assert d["steps"] == 20 and d["warmup"] == 5
    # only the contract's fields travel in the line; the long ones stay in the detail
    assert "path" not in d["e2e"] and "single_thread" not in d["cpu_baseline"]


def test_headline_without_cpu_baseline_still_parses():
    d = json.loads(_fake_headline(cpu=None))
    assert d["cpu_baseline"] is None


@pytest.mark.parametrize("n", [1, 5, 20, 63, 64, 65, 128, 130, 2000, 20000])
def test_replay_plan_covers_exactly_n_steps(n):
    rem, full = bench.replay_plan(n, 64)
    assert 0 <= rem < 64 and rem + 64 * full == n


def test_reference_arm_line_is_small_and_complete():
    # the reference arm times the float64 oracle on the host: run it for one
    # tiny step and check the line it prints
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.strip().splitlines()
    assert len(lines) == 1 and len(lines[0]) <= MAX_LINE
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
