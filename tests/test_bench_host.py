"""Host-side pieces of bench.py that need no GPU: the algorithmic work
model, the per-path arithmetic type, and the reference arm of the stage in
front of the memory (the oracle on host cores)."""
import json
import os
import subprocess
import sys

import pytest

import bench
from harness import PROLOGUES, WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_path_dtype_names_each_path():
    assert bench.path_dtype(WORKLOADS["titans_mlp"]) == "bf16"          # fused MLP kernel
    assert bench.path_dtype(WORKLOADS["titans_chunkwise"]) == "bf16"
    assert bench.path_dtype(WORKLOADS["atlas_muon"]) == "bf16x3"        # split-bf16 Newton-Schulz
    assert bench.path_dtype(WORKLOADS["atlas_long"]) == "bf16x3"
    for name in ("linear_f32", "atlas_poly_c4", "atlas_poly_c16", "atlas_muon_surprise"):
        assert bench.path_dtype(WORKLOADS[name]) == "f32", name


def test_chunkwise_work_is_below_the_per_token_work():
    """One update per chunk: the chunk-wise rule's algorithmic FLOPs are
    below the per-token rule's on the same geometry, and with Muon the
    Newton-Schulz share drops by about the chunk length."""
    t, tc = WORKLOADS["titans_mlp"], WORKLOADS["titans_chunkwise"]
    assert bench.flops_per_chunk(tc) < bench.flops_per_chunk(t)
    m, mc = WORKLOADS["atlas_muon"], WORKLOADS["atlas_muon_chunkwise"]
    ratio = bench.flops_per_chunk(m) / bench.flops_per_chunk(mc)
    assert 30 < ratio < 64


def test_prologue_bytes_per_step():
    p = PROLOGUES["titans_prologue"]
    # x (bf16) + W_in (bf16) + taps and biases (fp32) in; q, k, v (bf16) and 3 gates (fp32) out
    want = (16384 * 512 * 2 + 512 * 1560 * 2 + 4 * (1536 * 4 + 3 * 8)
            + 16384 * 8 * (2 * 192 + 4 * 3))
    assert bench.prologue_bytes_per_step(p) == want


def test_prologue_reference_arm_runs_the_oracle_on_host_cores():
    r = subprocess.run([sys.executable, "bench.py", "--workload", "small_prologue_f32", "--impl", "reference"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == "small_prologue_f32"


def test_every_named_workload_is_a_bench_choice():
    with pytest.raises(SystemExit):
        bench.main(["--workload", "no_such_workload"])
