"""The benchmark's own bookkeeping, on CPU.

Every committed ncu summary names the kernel sources it was taken on (a
sha256 prefix); the bench reports a summary's DRAM traffic only while the
sources still match, so a kernel edited after its capture must be captured
again.  These tests check that the summaries the default run reads match
the current sources, and that the reference arm (the oracle on the host
cores) prints the contract's JSON line.
"""
import json
import os
import re
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _summary_sources(name):
    """(kernel, pool element type) whose sources a summary file covers."""
    dtype = "bf16" if name.endswith("_bf16.md") else "fp8" if name.endswith("_fp8.md") else "f32"
    if name.startswith("decode_"):
        return "decode", dtype
    if name.startswith("prefill_tc_") or name.startswith("split_"):
        return "prefill", dtype
    raise AssertionError("unknown summary " + name)


@pytest.mark.parametrize("name", sorted(f for f in os.listdir(PROFILES) if f.endswith(".md")))
def test_summary_taken_on_current_sources(name):
    text = open(os.path.join(PROFILES, name)).read()
    m = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    assert m, name + " names no source digest"
    kernel, dtype = _summary_sources(name)
    assert m.group(1) == bench.kernel_source_digest(kernel, dtype), (
        name + " was taken on other kernel sources: capture it again")


@pytest.mark.parametrize("workload,kernel,dtype", [
    ("continuous_batching_m256", "decode", "f32"),
    ("batched_decode_m64", "decode", "f32"),
    ("continuous_batching_small", "decode", "f32"),
    ("continuous_batching_m256", "decode", "bf16"),
    ("continuous_batching_m256", "decode", "fp8"),
    ("chunked_prefill", "prefill", "f32"),
    ("chunked_prefill", "prefill", "bf16"),
    ("shared_prefix_forks", "prefill", "f32"),
])
def test_traffic_lookups_resolve(workload, kernel, dtype):
    t = bench.profiled_traffic(workload, kernel, dtype)
    assert t is not None and t > 0


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        "continuous_batching_small", "--steps", "1", "--warmup", "3", "--cpu-budget", "0.3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "continuous_batching_small"
    assert d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
