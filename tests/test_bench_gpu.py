"""The benchmark's own arm on a GPU: one JSON line with the keys of the contract.

Runs `bench.py` on the MoE-shaped K = 7168 workload with few steps and checks the line's
structure and its internal consistency: the value and the step time agree, the roofline
fraction is the algorithmic bytes over the value against the peak, the end-to-end number
declares the bytes it copies, one launch of this library per timed call, the clock record is
not empty, and the prepack and cold-call legs are present. Values are not compared with any
target (that is the benchmark's job), only checked to be positive and finite.
"""
import json
import math
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "20", "--warmup", "3",
                        "--no-cpu-baseline", "--no-other-workloads", "--e2e-steps", "3"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def positive(x):
    return isinstance(x, (int, float)) and math.isfinite(x) and x > 0


def test_headline_keys(line):
    for k in ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"]:
        assert k in line, k
    assert line["unit"] == "us" and line["higher_is_better"] is False and line["n_gpus"] == 1
    assert line["steps"] == 20 and line["warmup"] == 3
    assert line["config"]["workload"] == "moe_g8_n4096_k7168"
    assert positive(line["value"]) and abs(line["ms_per_step"] * 1e3 - line["value"]) < 1e-2


def test_roofline_is_the_algorithmic_bytes_over_the_value(line):
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and positive(rf["peak"])
    gbs = rf["algorithmic_bytes_per_launch"] / (line["value"] * 1e-6) / 1e9
    assert abs(gbs - rf["achieved"]) / gbs < 0.01
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert rf["traffic"] is None or positive(rf["traffic"])


def test_end_to_end_declares_its_copies(line):
    e = line["e2e"]
    assert positive(e["value"]) and e["unit"] == "us"
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    # the host copies make a step slower than the device-resident call
    assert e["value"] > line["value"]


def test_one_launch_per_call_and_a_clock_record(line):
    assert line["gpu_launches"] == line["steps"]  # prepacked scales: one kernel a call
    c = line["clocks"]
    assert c["samples"] > 0 and positive(c["sm_mhz"]) and positive(c["sm_max_mhz"])


def test_prepack_and_cold_call_legs(line):
    p = line["prepack"]
    assert positive(p["value"]) and positive(p["chained"]["value"]) and positive(p["flushed_floor_us"])
    assert p["algorithmic_bytes"] == p["read_bytes"] + p["written_bytes"]
    cc = line["cold_call"]
    assert positive(cc["miss"]["gpu_us"]) and positive(cc["hit"]["gpu_us"])


@pytest.mark.parametrize("split", ["groups", "n"])
def test_split_modes_run_at_one_rank(split):
    # --split shards one call across the ranks; with one rank the share is the whole call,
    # and the line says so (strong scaling, the sharding in `parallelism`)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "10", "--warmup", "3", "--split", split,
                        "--no-cpu-baseline", "--no-other-workloads", "--e2e-steps", "2"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["scaling"] == "strong" and split in d["config"]["parallelism"]
    assert positive(d["value"]) and d["config"]["workload"] == "moe_g8_n4096_k7168"
