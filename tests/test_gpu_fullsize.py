"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (every unit, every token, one call), on outputs the oracle can compute
one by one:

* prefix: the first chunks of sampled units, from the true initial state;
* last chunk: sampled units' last chunk recomputed by the oracle from the
  library's own state after T - C tokens (a second call), compared with the
  full call's last-chunk read-out and final W, S (this also checks that one
  call equals two chained calls at full size).
"""
import numpy as np
import pytest

import oracle
from harness import WORKLOADS, bf16_from_bits, make_inputs
from tests.gpu_common import TOL, flat_units, maxrel

pytestmark = pytest.mark.gpu

SEQ = ("q", "k", "v", "theta", "eta", "alpha", "gamma")


def _run(w, t, T=None, win=None):
    import torch
    from test_learned_neural_gb300.runner import Memory
    mem = Memory(w)
    if T is not None:
        t = {k: (v[:, :, :T].contiguous() if k in SEQ and v is not None else v) for k, v in t.items()}
    out = mem.forward(t, win=win)
    torch.cuda.synchronize()
    mem.status()
    res = {"y": out["y"].cpu().numpy(), "W": [m.cpu().numpy() for m in out["W"]],
           "S": [m.cpu().numpy() for m in out["S"]]}
    for key in ("win_k", "win_v", "win_gamma"):
        if key in out:
            res[key] = out[key].cpu()
    mem.close()
    return res


def _sample_units(w):
    return sorted({0, w.units - 1})


@pytest.mark.parametrize("name", ["titans_mlp", "atlas_muon", "atlas_long", "atlas_poly_c4", "atlas_poly_c16",
                                  "atlas_muon_surprise", "titans_chunkwise", "atlas_muon_chunkwise"])
def test_full_size_prefix(gpu_lib, name):
    from test_learned_neural_gb300.runner import tensors_from_numpy
    w = WORKLOADS[name]
    inp = make_inputs(w)
    g = _run(w, tensors_from_numpy(inp))
    T0 = 2 * w.C
    units = _sample_units(w)
    r = oracle.forward(w, inp, units=units, T=T0)
    err = maxrel(flat_units(g["y"])[units][:, :T0], r["y"])
    print(name, "prefix y", f"{err:.2e}")
    assert err <= TOL[w.qkv_dtype]


def _to64(t, dtype):
    import torch
    a = t.numpy() if t.dtype != torch.bfloat16 else t.view(torch.int16).numpy().view(np.uint16)
    return bf16_from_bits(a).astype(np.float64) if dtype == "bf16" else a.astype(np.float64)


@pytest.mark.parametrize("name", ["titans_mlp", "atlas_muon", "atlas_long", "titans_chunkwise",
                                  "atlas_muon_chunkwise"])
def test_full_size_last_chunk(gpu_lib, name):
    from test_learned_neural_gb300.runner import tensors_from_numpy
    w = WORKLOADS[name]
    inp = make_inputs(w)
    t = tensors_from_numpy(inp)
    full = _run(w, t)
    head = _run(w, t, T=w.T - w.C)
    units = _sample_units(w)
    s = w.T - w.C
    for u in units:
        d = oracle.unit_inputs(w, inp, u)
        cache = None
        if w.c > 1:
            cache = (_to64(head["win_k"].reshape(w.units, w.c - 1, w.d_k)[u], w.qkv_dtype),
                     _to64(head["win_v"].reshape(w.units, w.c - 1, w.d_v)[u], w.qkv_dtype),
                     head["win_gamma"].reshape(w.units, w.c - 1)[u].numpy().astype(np.float64))
        W0 = [flat_units(m)[u] for m in head["W"]]
        S0 = [flat_units(m)[u] for m in head["S"]]
        kw = {} if cache is None else dict(cache_k=cache[0], cache_v=cache[1], cache_g=cache[2])
        y, W, S, _ = oracle.forward_unit(
            w, d["k"][s:], d["q"][s:], d["v"][s:], d["theta"][s:], d["eta"][s:], d["alpha"][s:],
            None if d["gamma"] is None else d["gamma"][s:], W0, S0, d["P"], **kw)
        ey = maxrel(flat_units(full["y"])[u][s:], y)
        eW = max(maxrel(flat_units(full["W"][m])[u], W[m]) for m in range(len(W)))
        eS = max(maxrel(flat_units(full["S"][m])[u], S[m]) for m in range(len(S)))
        print(name, "unit", u, f"last chunk y {ey:.2e}  W {eW:.2e}  S {eS:.2e}")
        assert ey <= TOL[w.qkv_dtype] and eW <= TOL[w.qkv_dtype] and eS <= 5 * TOL[w.qkv_dtype]
