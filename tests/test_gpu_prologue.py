"""CUDA stage in front of the memory (projection, short causal convolution,
q/k normalisation, gate heads) vs its fp64 oracle on the same seeded inputs,
element by element; and the stage chained into the memory forward."""
import numpy as np
import pytest

import oracle
from harness import PROLOGUES, WORKLOADS, bf16_bits, bf16_from_bits, make_inputs, make_prologue_inputs
from tests.gpu_common import TOL, maxrel

pytestmark = pytest.mark.gpu

OUTS = ("q", "k", "v", "theta", "eta", "alpha", "gamma")
# q, k, v are stored in the input type (bf16 rounding: 2^-9 relative); the
# gates and the carried cache are fp32 from an fp32-accumulated projection
QKV_TOL = {"f32": 1e-4, "bf16": 1e-2}
F32_TOL = 1e-4


def _decode(a, dtype):
    if a is None:
        return None
    return bf16_from_bits(a).astype(np.float64) if dtype == "bf16" else np.asarray(a, np.float64)


def _host(t):
    import torch
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return bf16_from_bits(t.cpu().view(torch.int16).numpy().view(np.uint16)).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def _oracle_rows(p, inp, rows=None, t0=0, t1=None):
    """Oracle outputs of the listed batch rows on tokens [t0, t1)."""
    rows = range(p.B) if rows is None else rows
    x = _decode(inp["x"], p.qkv_dtype)
    W = _decode(inp["W_in"], p.qkv_dtype)
    res = []
    for b in rows:
        cache = None if inp["cache"] is None or t0 > 0 else inp["cache"][b]
        res.append(oracle.prologue_row(p, x[b, t0:t1], W, inp["conv_w"], inp["gate_b"], cache))
    return res


def _run(p, inp, T=None):
    import torch
    from test_learned_neural_gb300.runner import Prologue, prologue_tensors_from_numpy
    pro = Prologue(p)
    t = prologue_tensors_from_numpy(inp)
    if T is not None:
        t["x"] = t["x"][:, :T].contiguous()
    out = pro.forward(t)
    torch.cuda.synchronize()
    pro.status()
    res = {k: _host(v) for k, v in out.items()}
    res["_gemm"] = pro.last_gemm()
    pro.close()
    return res


def _tensor_core_projection(p):
    """The projection runs on the tensor cores (TMA-fed tcgen05 tiles) for
    bf16 inputs whose row strides TMA can take (D and N multiples of 8)."""
    return p.qkv_dtype == "bf16" and p.D % 8 == 0 and p.N % 8 == 0


def _check(p, g, ref, rows, sl=slice(None), cache=True):
    for key in OUTS:
        if ref[0][key] is None:
            assert key not in g
            continue
        want = np.stack([r[key] for r in ref])
        got = g[key][rows][:, :, sl]
        tol = QKV_TOL[p.qkv_dtype] if key in ("q", "k", "v") else F32_TOL
        err = maxrel(got, want[:, :, sl])
        print(p.name, key, f"{err:.2e}")
        assert err <= tol, (key, err)
    if cache and p.conv > 1:
        err = maxrel(g["cache"][rows], np.stack([r["cache"] for r in ref]))
        assert err <= F32_TOL, ("cache", err)


SMALL = [
    ("titans_prologue", dict(B=1, T=100)),        # 8 heads of 64; 100 = a 64-token tile + a ragged 36
    ("atlas_prologue", dict(B=2, T=70)),          # 16 heads of 48, gamma head
    ("small_prologue_f32", dict()),               # fp32, widths 8 and 12, 40-wide model
    ("small_prologue_f32", dict(conv=1)),         # no convolution
    ("small_prologue_f32", dict(conv=8, T=5)),    # more taps than tokens
    ("small_prologue_f32", dict(d_k=7, d_v=5)),   # odd widths: single channels, 4-byte copies
    ("atlas_prologue", dict(B=1, T=40, D=50, H=3, d_k=9, d_v=6)),   # bf16, odd q/k width
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c[0] + "-" + "-".join(f"{k}{v}" for k, v in c[1].items()))
@pytest.mark.parametrize("with_cache", [False, True])
def test_small_parity(gpu_lib, case, with_cache):
    name, kw = case
    p = PROLOGUES[name].scaled(**kw)
    inp = make_prologue_inputs(p, cache=with_cache and p.conv > 1)
    g = _run(p, inp)
    assert g["_gemm"] == (1 if _tensor_core_projection(p) else 0)
    _check(p, g, _oracle_rows(p, inp), list(range(p.B)))


def test_split_calls_carry_the_cache(gpu_lib):
    """Two calls chained through cache_out equal one call (to the GEMM's
    accumulation order), also when the first call is shorter than the
    cache."""
    import torch
    from test_learned_neural_gb300.runner import Prologue, prologue_tensors_from_numpy
    p = PROLOGUES["small_prologue_f32"].scaled(T=40)
    inp = make_prologue_inputs(p, cache=True)
    pro = Prologue(p)
    t = prologue_tensors_from_numpy(inp)
    whole = pro.forward(t)
    for T1 in (2, 17):
        a = pro.forward(dict(t, x=t["x"][:, :T1].contiguous()))
        b = pro.forward(dict(t, x=t["x"][:, T1:].contiguous(), cache=a["cache"].clone()))
        torch.cuda.synchronize()
        for key in OUTS:
            if key in whole:
                joined = torch.cat([a[key], b[key]], dim=2)
                err = maxrel(_host(joined), _host(whole[key]))
                assert err <= 1e-5, (T1, key, err)
        assert maxrel(_host(b["cache"]), _host(whole["cache"])) <= 1e-5
    pro.close()


@pytest.mark.parametrize("name", ["titans_prologue", "atlas_prologue"])
def test_full_size_sampled(gpu_lib, name):
    """Full size, one launch pair as bench.py times it: the first 96 tokens
    and the last 64 of the first and last batch rows against the oracle (the
    last window recomputed from the three tokens before it)."""
    p = PROLOGUES[name]
    inp = make_prologue_inputs(p)
    g = _run(p, inp)
    assert g["_gemm"] == 1
    rows = sorted({0, p.B - 1})
    _check(p, g, _oracle_rows(p, inp, rows, 0, 96), rows, slice(0, 96), cache=False)
    K = p.conv
    tail = _oracle_rows(p, inp, rows, p.T - 64 - (K - 1), p.T)
    for key in OUTS:
        if tail[0][key] is None:
            continue
        want = np.stack([r[key][:, K - 1:] for r in tail])
        err = maxrel(g[key][rows][:, :, p.T - 64:], want)
        tol = QKV_TOL[p.qkv_dtype] if key in ("q", "k", "v") else F32_TOL
        assert err <= tol, (key, err)
    want = np.stack([r["cache"] for r in tail])
    assert maxrel(g["cache"][rows], want) <= F32_TOL


def test_chained_into_the_memory(gpu_lib):
    """x -> stage -> memory forward on the GPU against the two oracles
    chained (the stage's fp64 q, k, v rounded to the memory's bf16 inputs)."""
    import torch
    from test_learned_neural_gb300.runner import Memory, Prologue, prologue_tensors_from_numpy, tensors_from_numpy
    w = WORKLOADS["titans_mlp"].scaled(B=1, H=2, T=128)
    p = PROLOGUES["titans_prologue"].scaled(B=1, H=2, D=128, T=128)
    pin = make_prologue_inputs(p)
    mem_in = make_inputs(w)                  # W0, S0 of the memory
    pro = Prologue(p)
    st = pro.forward(prologue_tensors_from_numpy(pin))
    t = tensors_from_numpy(mem_in)
    for key in ("q", "k", "v", "theta", "eta", "alpha"):
        t[key] = st[key]
    mem = Memory(w)
    out = mem.forward(t)
    torch.cuda.synchronize()
    mem.status()
    ref = _oracle_rows(p, pin)[0]
    chained = dict(mem_in)
    for key in ("q", "k", "v"):
        chained[key] = bf16_bits(ref[key][None])          # [1, H, T, d] as the memory's bf16 input
    for key in ("theta", "eta", "alpha"):
        chained[key] = ref[key][None].astype(np.float32)
    r = oracle.forward(w, chained)
    err = maxrel(_host(out["y"]).reshape(r["y"].shape), r["y"])
    errW = max(maxrel(_host(out["W"][m]).reshape(r["W"][m].shape), r["W"][m]) for m in range(2))
    print("chained y", f"{err:.2e}", "W", f"{errW:.2e}")
    assert err <= TOL["bf16"] and errW <= TOL["bf16"]
    pro.close()
    mem.close()
