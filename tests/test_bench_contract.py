"""The JSON line of bench.py's reference arm (the fp64 oracle on the host cores) and the
CPU-baseline record, checked on CPU: the keys the benchmark contract names, the same
config as the GPU arm, and no host-device bytes for a host-only run."""
import json
import subprocess
import sys
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                          "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600, check=True)
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["higher_is_better"] is True and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    import bench
    from expert_gemm_gb300 import workloads as W
    assert d["config"] == bench.workload_config(W.get("tiny"), 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and 1 <= cb["cores"] <= cb["host_cores"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_cpu_baseline_all_cores_and_one():
    import bench
    from expert_gemm_gb300 import workloads as W
    wl = W.get("tiny")
    cb = bench.cpu_baseline(wl, 0.3)
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s" and cb["value"] > 0
    assert 1 <= cb["cores"] <= min(cb["host_cores"], 16)
    assert cb["one_core"]["cores"] == 1 and cb["one_core"]["value"] > 0


@pytest.mark.parametrize("warmup", ["0", "2"])
def test_too_few_warmup_steps_refused(warmup):
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                          "--warmup", warmup], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode != 0 and "warmup" in out.stderr


def test_secondary_legs_are_long_enough_to_sample_clocks():
    """Each secondary configuration times ~0.6 s of steps (the clock sampler polls every
    200 ms), never fewer than the headline's steps, and reports its step in SM cycles."""
    import bench
    assert bench.secondary_steps(0.06, 20) == 4615          # one-token layer
    assert bench.secondary_steps(3.6, 20) == 163             # prefill
    assert bench.secondary_steps(3.6, 500) == 500
    assert bench.secondary_steps(100.0, 3) == 10
    assert set(bench.SECONDARY) == {"prefill", "wide", "sweep_T1", "sweep_T16", "sweep_T256", "sweep_T4096",
                                    "dense_decode"}
    c = bench.clock_summary({"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}, 0.5)
    assert c["kcycles_per_step"] == 1000.0 and c["samples"] == 3
    assert bench.clock_summary(None, 1.0) is None
