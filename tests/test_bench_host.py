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
    for name in ("atlas_poly_c4", "atlas_poly_c16"):                     # split-bf16 depth-1 kernel
        assert bench.path_dtype(WORKLOADS[name]) == "bf16x3", name
    assert bench.path_dtype(WORKLOADS["atlas_muon_surprise"]) == "bf16x3"   # tensor-core read-out and state
    assert bench.path_dtype(WORKLOADS["linear_f32"]) == "f32"


def test_chunkwise_work_is_below_the_per_token_work():
    """One update per chunk: the chunk-wise rule's algorithmic FLOPs are
    below the per-token rule's on the same geometry, and with Muon the
    Newton-Schulz share drops by about the chunk length."""
    t, tc = WORKLOADS["titans_mlp"], WORKLOADS["titans_chunkwise"]
    assert bench.flops_per_chunk(tc) < bench.flops_per_chunk(t)
    m, mc = WORKLOADS["atlas_muon"], WORKLOADS["atlas_muon_chunkwise"]
    ratio = bench.flops_per_chunk(m) / bench.flops_per_chunk(mc)
    assert 30 < ratio < 64


def test_algorithmic_flops_follow_the_scope_table():
    """Per-token FLOPs by the hot-path scope table's accounting: config 3
    (Muon, 128 x 512 matrices, five steps) 2 x 5 x (2 * 128^2 * 512 * 2 +
    2 * 128^3) = 377 M; config 4 = Newton-Schulz on 64 x 256 plus phi P
    (2 x 2145 x 64 per key and per query) = 47.8 M; config 1 ~0.35 M;
    config 2 the table's items phi(k) W_bar 72 k + S/W updates 144 k +
    phi(q) W_bar/S_bar 144 k + intra-chunk Gram 72-89 k = 432-449 k (the
    table's rounded total, 0.37-0.40 M, is below its own items); config 0
    ~10 k."""
    f = bench.algorithmic_flops_per_token
    assert f(WORKLOADS["atlas_muon"]) == 2 * 5 * (2 * 128 ** 2 * 512 * 2 + 2 * 128 ** 3) == 377487360
    assert abs(f(WORKLOADS["atlas_long"]) - 47.8e6) < 0.1e6
    assert 0.34e6 < f(WORKLOADS["titans_mlp"]) < 0.37e6
    assert 0.43e6 < f(WORKLOADS["atlas_poly_c4"]) < f(WORKLOADS["atlas_poly_c16"]) < 0.45e6
    assert 9e3 < f(WORKLOADS["linear_f32"]) < 12e3


def test_roofline_bound_from_intensity():
    peaks = {"bf16_tflops_sustained": 1737.5, "hbm_gbs": 6705.2}
    w = WORKLOADS["atlas_muon"]
    fl = bench.algorithmic_flops_per_token(w) * w.tokens
    assert bench.roofline_bound(w, fl, bench.bytes_per_step(w), peaks) == "tensor"
    assert bench.roofline_bound(w, 1.0, 1e9, peaks) == "hbm"
    assert bench.roofline_bound(WORKLOADS["linear_f32"], 1e12, 1.0, peaks) == "alu"   # fp32 SIMT path
    # the polynomial workloads run the split-bf16 tensor-core kernel
    wp = WORKLOADS["atlas_poly_c4"]
    assert bench.path_dtype(wp) == "bf16x3"
    fl = bench.algorithmic_flops_per_token(wp) * wp.tokens
    assert bench.roofline_bound(wp, fl, bench.bytes_per_step(wp), peaks) == "tensor"
    assert bench.path_dtype(wp.scaled(qkv_dtype="f32")) == "f32"


def test_reference_sample_is_bounded():
    """The reference arm's per-step sample shrinks with the step count, so
    K steps take about a minute of oracle work, never below 8 tokens."""
    w = WORKLOADS["atlas_muon"]
    units, T = bench.oracle_sample(w, budget_s=60.0 / 100)
    assert 8 <= T <= 2 * w.C and T * bench.ORACLE_S_PER_TOKEN["atlas_muon"] <= 0.61
    units, T10 = bench.oracle_sample(w, budget_s=6.0)
    assert T10 == 2 * w.C
    assert bench.default_steps("atlas_muon") == 10 and bench.default_steps("titans_mlp") == 100


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
