"""CUDA library vs the fp64 oracle on the same seeded inputs, element by
element, at sizes the oracle finishes in seconds (several chunks each)."""
import numpy as np
import pytest

import oracle
from harness import WORKLOADS, make_inputs
from tests.gpu_common import TOL, compare, flat_units, maxrel, run_gpu

pytestmark = pytest.mark.gpu

SMALL = {
    "linear_f32": dict(),                         # full size: 1 unit x 256 tokens
    "titans_mlp": dict(B=1, H=2, T=256),
    "atlas_poly_c4": dict(B=1, H=2, T=256),
    "atlas_poly_c16": dict(B=1, H=2, T=256),
    "atlas_muon": dict(B=1, H=1, T=128),
    "atlas_long": dict(B=1, H=2, T=192),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_parity(gpu_lib, name):
    w = WORKLOADS[name].scaled(**SMALL[name]) if SMALL[name] else WORKLOADS[name]
    errs = compare(w)
    tol = TOL[w.qkv_dtype]
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["y"] <= tol
    for k, v in errs.items():
        if k.startswith("W"):
            assert v <= tol, (k, v)
        if k.startswith("S"):
            assert v <= 5 * tol, (k, v)


@pytest.mark.parametrize("name", list(SMALL))
def test_small_parity_pre_update_readout(gpu_lib, name):
    """Read-out with the memory before each token's update (titans-pytorch-mlx
    README, MAC, Eq. 21) on every path: fused MLP kernel, depth-1 split path,
    tensor-core Newton-Schulz with its decay scans."""
    w = (WORKLOADS[name].scaled(**SMALL[name]) if SMALL[name] else WORKLOADS[name]).scaled(readout="pre")
    errs = compare(w)
    tol = TOL[w.qkv_dtype]
    print(name, "pre", {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["y"] <= tol
    for k, v in errs.items():
        if k.startswith("W"):
            assert v <= tol, (k, v)
        if k.startswith("S"):
            assert v <= 5 * tol, (k, v)


@pytest.mark.parametrize("name", ["titans_mlp", "atlas_poly_c16", "atlas_long"])
def test_split_continuation_matches_whole(gpu_lib, name):
    """Two calls with carried W, S and window cache equal one call."""
    import torch
    from test_learned_neural_gb300.runner import Memory, tensors_from_numpy
    w = WORKLOADS[name].scaled(B=1, H=2, T=256)
    inp = make_inputs(w)
    whole = run_gpu(w, inp)
    mem = Memory(w)
    t = tensors_from_numpy(inp)
    T1 = 128
    first = {k: (v[:, :, :T1].contiguous() if k in ("q", "k", "v", "theta", "eta", "alpha", "gamma")
                 and v is not None else v) for k, v in t.items()}
    o1 = mem.forward(first)
    second = {k: (v[:, :, T1:].contiguous() if k in ("q", "k", "v", "theta", "eta", "alpha", "gamma")
                  and v is not None else v) for k, v in t.items()}
    second["W0"], second["S0"] = o1["W"], o1["S"]
    win = None
    if w.c > 1:
        win = (w.c - 1, o1["win_k"], o1["win_v"], o1["win_gamma"])
    o2 = mem.forward(second, win=win)
    torch.cuda.synchronize()
    y = np.concatenate([o1["y"].cpu().numpy(), o2["y"].cpu().numpy()], axis=2)
    assert maxrel(y, whole["y"]) < 1e-5
    for m in range(len(o2["W"])):
        assert maxrel(o2["W"][m].cpu().numpy(), whole["W"][m]) < 1e-5
    mem.close()


@pytest.mark.parametrize("H,T", [(2, 128), (4, 256), (3, 512)])
def test_host_buffers_match_device_buffers(gpu_lib, H, T):
    """Host-buffer entry point = device entry point, bit for bit.  With T a
    multiple of four chunks the fused path's host call runs pipelined over
    four time segments (one launch each, the state handed on in fp32)."""
    w = WORKLOADS["titans_mlp"].scaled(B=1, H=H, T=T)
    inp = make_inputs(w)
    d = run_gpu(w, inp)
    h = run_gpu(w, inp, host=True)
    np.testing.assert_array_equal(d["y"], h["y"])
    for m in range(2):
        np.testing.assert_array_equal(d["W"][m], h["W"][m])


def test_window_cache_out_holds_the_last_tokens(gpu_lib):
    w = WORKLOADS["atlas_poly_c4"].scaled(B=1, H=2, T=128)
    inp = make_inputs(w)
    g = run_gpu(w, inp)
    k = flat_units(inp["k"])[:, -(w.c - 1):]
    got = g["win_k"].view(-1, w.c - 1, w.d_k).view(dtype=__import__("torch").int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, k)
    np.testing.assert_array_equal(g["win_gamma"].numpy().reshape(-1, w.c - 1), flat_units(inp["gamma"])[:, -(w.c - 1):])


def test_alpha_one_wipes_state_on_gpu(gpu_lib):
    """alpha = 1: the final W equals the final (orthogonalised) momentum."""
    w = WORKLOADS["atlas_long"].scaled(B=1, H=1, T=64)
    inp = make_inputs(w)
    inp["alpha"] = np.ones_like(inp["alpha"])
    g = run_gpu(w, inp)
    S = g["S"]
    for m in range(2):
        U = oracle.newton_schulz(flat_units(S[m])[0], w.ns_iters)
        assert maxrel(flat_units(g["W"][m])[0], U) < 2e-3


@pytest.mark.parametrize("readout", ["post", "pre"])
def test_streaming_one_token_calls(gpu_lib, readout):
    """Streaming decode: with one-token chunks (C = 1) a sequence fed one
    token per call, carrying W, S and the Omega window cache between calls,
    equals one call over the whole sequence and the oracle."""
    import torch
    from test_learned_neural_gb300.runner import Memory, tensors_from_numpy
    w = WORKLOADS["atlas_poly_c4"].scaled(B=1, H=2, T=12, C=1, readout=readout)
    inp = make_inputs(w)
    whole = run_gpu(w, inp)
    r = oracle.forward(w, inp)
    assert maxrel(flat_units(whole["y"]), r["y"]) <= TOL[w.qkv_dtype]
    mem = Memory(w)
    t = tensors_from_numpy(inp)
    seq = ("q", "k", "v", "theta", "eta", "alpha", "gamma")
    W, S, win, ys = t["W0"], t["S0"], None, []
    for i in range(w.T):
        step = {k: (v[:, :, i:i + 1].contiguous() if k in seq and v is not None else v) for k, v in t.items()}
        step["W0"], step["S0"] = W, S
        o = mem.forward(step, win=win)
        ys.append(o["y"].cpu().numpy())
        W, S = o["W"], o["S"]
        win = (min(w.c - 1, i + 1), o["win_k"], o["win_v"], o["win_gamma"])
    torch.cuda.synchronize()
    mem.status()
    y = np.concatenate(ys, axis=2)
    assert maxrel(y, whole["y"]) < 1e-5
    for m in range(len(W)):
        assert maxrel(W[m].cpu().numpy(), whole["W"][m]) < 1e-5
    mem.close()


SURPRISE = {
    "linear_f32": dict(ns_iters=5, c=3),                       # fp32, Omega window 3
    "atlas_poly_c4": dict(B=1, H=2, T=256, ns_iters=5),        # depth 1, degree-2 features
    "titans_mlp": dict(B=1, H=2, T=256, ns_iters=5),           # c = 1: rank-one surprise
    "atlas_muon_surprise": dict(B=1, H=1, T=128),              # 128 -> 512 -> 128, c = 8
    "atlas_long": dict(B=1, H=2, T=192),                       # projected features, c = 8
}


@pytest.mark.parametrize("name", list(SURPRISE))
@pytest.mark.parametrize("readout", ["post", "pre"])
def test_small_parity_surprise_ns(gpu_lib, name, readout):
    """Newton-Schulz on each token's windowed surprise (atlas-torch README,
    "Atlas Extensions"), run on the GPU as a c x c core iteration with banded
    dual-form coefficients, against the oracle's dense NS of g_t."""
    w = WORKLOADS[name].scaled(ns_target="surprise", readout=readout, **SURPRISE[name])
    errs = compare(w)
    tol = TOL[w.qkv_dtype]
    print(name, "surprise", readout, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["y"] <= tol
    for k, v in errs.items():
        if k.startswith("W"):
            assert v <= tol, (k, v)
        if k.startswith("S"):
            assert v <= 5 * tol, (k, v)


SURPRISE_TC_RAGGED = [
    ("C48_c16", dict(B=1, H=1, T=96, C=48, c=16)),          # 48-token chunks (rows 48-63 of the tiles empty), 63 window rows
    ("C16_c1", dict(B=1, H=2, T=64, C=16, c=1)),            # short chunks, rank-one surprise
]


@pytest.mark.parametrize("case", SURPRISE_TC_RAGGED, ids=[c[0] for c in SURPRISE_TC_RAGGED])
@pytest.mark.parametrize("readout", ["post", "pre"])
def test_surprise_tensor_core_path_ragged_chunks(gpu_lib, case, readout):
    """The tensor-core surprise read-out and state (per-unit band products
    in 16-token groups, column-block read-outs) on chunks shorter than the
    64-row tiles and on the widest window they take (atlas-torch README,
    "Atlas Extensions": Newton-Schulz of the surprise over the Omega window)."""
    _, kw = case
    w = WORKLOADS["atlas_muon_surprise"].scaled(readout=readout, **kw)
    errs = compare(w)
    tol = TOL[w.qkv_dtype]
    print(case[0], readout, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["y"] <= tol
    for k, v in errs.items():
        if k.startswith("W"):
            assert v <= tol, (k, v)
        if k.startswith("S"):
            assert v <= 5 * tol, (k, v)


@pytest.mark.parametrize("name", ["atlas_poly_c4", "atlas_long", "atlas_muon_surprise"])
def test_repeated_calls_replay_identically(gpu_lib, name):
    """Identical repeated calls replay a captured CUDA graph of the launch
    sequence: its results equal a direct run's bit for bit, and new data in
    the same buffers is read."""
    import torch
    from test_learned_neural_gb300.runner import Memory, tensors_from_numpy
    w = WORKLOADS[name].scaled(B=1, H=2, T=128)
    inp = make_inputs(w)
    mem = Memory(w)
    t = tensors_from_numpy(inp)
    out = mem.alloc_outputs(w.B, w.H, w.T, "cuda")
    results = []
    for _ in range(4):                       # direct, capture, replay, replay
        mem.forward(t, out=out)
        torch.cuda.synchronize()
        results.append(out["y"].clone())
    mem.status()
    for r in results[1:]:
        assert torch.equal(r, results[0])
    with torch.no_grad():
        t["q"].mul_(0.5)                     # new data, same buffer: replayed
    mem.forward(t, out=out)
    torch.cuda.synchronize()
    fresh = Memory(w)
    ref = fresh.forward(t)
    torch.cuda.synchronize()
    assert torch.equal(out["y"], ref["y"])
    for m in range(len(ref["W"])):
        assert torch.equal(out["W"][m], ref["W"][m])
    mem.close()
    fresh.close()


CHUNKWISE = [
    ("linear_f32", dict()),                                 # depth 1, fp32, 16 chunks
    ("linear_f32", dict(ns_iters=5)),                       # depth 1 with Muon (SIMT Newton-Schulz)
    ("titans_chunkwise", dict(B=1, H=2, T=256)),            # MLP 64 -> 256 -> 64
    ("atlas_poly_c4", dict(B=1, H=2, T=256, c=1)),          # degree-2 features (561 wide)
    ("atlas_muon_chunkwise", dict(B=1, H=1, T=128)),        # Muon on 128 x 512 (CTA-pair kernel)
    ("atlas_long", dict(B=1, H=2, T=192, c=1)),             # projected features, Muon short side 64
]


@pytest.mark.parametrize("case", CHUNKWISE, ids=lambda c: c[0] + ("_ns" if c[1].get("ns_iters") else ""))
@pytest.mark.parametrize("readout", ["post", "pre"])
def test_small_parity_chunkwise(gpu_lib, case, readout):
    """The titans-pytorch chunk-wise store path (atlas-torch README, "Bug
    Fixes": per_token_updates): one summed gradient, pooled gates and one
    momentum / decay step per chunk, Newton-Schulz once per chunk."""
    name, kw = case
    w = WORKLOADS[name].scaled(update="chunkwise", readout=readout, **kw)
    errs = compare(w)
    tol = TOL[w.qkv_dtype]
    print(name, "chunkwise", readout, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["y"] <= tol
    for k, v in errs.items():
        if k.startswith("W"):
            assert v <= tol, (k, v)
        if k.startswith("S"):
            assert v <= 5 * tol, (k, v)


def test_fused_kernel_reports_values_beyond_its_operand_range(gpu_lib):
    """The fused MLP kernel multiplies fp16 operands (scaled per tile by
    powers of two).  Values far beyond any normalised input (here v = 1e8,
    so dy leaves fp16's range and the outputs become non-finite) are
    reported as ATLAS_ERR_RANGE by the status call, without a fault; the
    next call on the same handle is valid."""
    import torch
    from test_learned_neural_gb300.runner import Memory, tensors_from_numpy
    from harness import bf16_bits
    w = WORKLOADS["titans_mlp"].scaled(B=1, H=2, T=128)
    inp = make_inputs(w)
    big = dict(inp)
    big["v"] = bf16_bits(np.full(inp["v"].shape, 1.0e8, np.float32))
    mem = Memory(w)
    mem.forward(tensors_from_numpy(big))
    torch.cuda.synchronize()
    assert gpu_lib.atlas_mem_status(mem.h) == gpu_lib.ATLAS_ERR_RANGE
    assert "non-finite" in gpu_lib.atlas_mem_last_error(mem.h)
    out = mem.forward(tensors_from_numpy(inp))
    torch.cuda.synchronize()
    assert gpu_lib.atlas_mem_status(mem.h) == gpu_lib.ATLAS_OK
    ref = oracle.forward(w, inp)
    assert maxrel(out["y"].cpu().numpy(), ref["y"]) <= TOL["bf16"]
    mem.close()
