"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (every unit, every token, one call), on outputs the oracle can compute
one by one:

* whole sequence: where the oracle runs a full-length unit in seconds (the
  Titans MLP memory, both update rules, and its slow-forgetting variant
  whose memory stays O(0.2) to the last token), every read-out and the
  final W, S of sampled units from the true initial state;
* prefix: the first chunks of sampled units, from the true initial state;
* restarts: sampled units' chunk at T/4, at T/2 and the last one,
  recomputed by the oracle from the library's own state at that token (a
  second, shorter call), compared with the full call's read-outs there;
  at the last chunk also with the final W, S.  Each restart also checks that
  one call equals two chained calls at full size (the recurrence is carried
  over chunk-by-chunk state and window cache only: titans-pytorch-mlx
  README, "Core Equations", Eq. 13-14; atlas-torch README, "Status and
  scope": chunked inference with carried state).
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


@pytest.mark.parametrize("name", ["titans_mlp", "titans_chunkwise", "titans_mlp_slow"])
def test_full_size_whole_sequence(gpu_lib, name):
    """Every token of y and the final W, S of two units over all T tokens,
    from W0 / S0, against the oracle run over the same whole sequence."""
    from test_learned_neural_gb300.runner import tensors_from_numpy
    w = WORKLOADS[name]
    inp = make_inputs(w)
    g = _run(w, tensors_from_numpy(inp))
    units = _sample_units(w)
    r = oracle.forward(w, inp, units=units)
    tol = TOL[w.qkv_dtype]
    ey = maxrel(flat_units(g["y"])[units], r["y"])
    # y of the slow-forgetting memory must differ from the queries late in
    # the sequence, or this comparison would not test the memory
    q_late = np.stack([oracle.unit_inputs(w, inp, u)["q"][-w.C:] for u in units])
    print(name, f"whole-sequence y {ey:.2e}", f"max|y - q| over the last chunk {np.abs(r['y'][:, -w.C:] - q_late).max():.2e}")
    assert ey <= tol
    for m in range(len(r["W"])):
        eW = maxrel(flat_units(g["W"][m])[units], r["W"][m])
        eS = maxrel(flat_units(g["S"][m])[units], r["S"][m])
        print(name, f"W{m} {eW:.2e}  S{m} {eS:.2e}")
        assert eW <= tol and eS <= 5 * tol
    if name == "titans_mlp_slow":
        assert np.abs(r["y"][:, -w.C:] - q_late).max() > 0.05
        assert min(np.abs(m).max() for m in r["W"]) > 0.05


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


_LAST = {}


def _full_call(name):
    """Inputs and the full-size call of one workload, kept for the next
    restart point of the same workload (one workload held at a time)."""
    from test_learned_neural_gb300.runner import tensors_from_numpy
    if name not in _LAST:
        _LAST.clear()
        w = WORKLOADS[name]
        inp = make_inputs(w)
        t = tensors_from_numpy(inp)
        _LAST[name] = (inp, t, _run(w, t))
    return _LAST[name]


RESTARTS = ["titans_mlp", "titans_mlp_slow", "atlas_muon", "atlas_long", "titans_chunkwise",
            "atlas_muon_chunkwise", "atlas_muon_surprise"]


@pytest.mark.parametrize("name,where", [(n, p) for n in RESTARTS for p in ("quarter", "half", "last")])
def test_full_size_restart(gpu_lib, name, where):
    """The full call's chunk at token s (T/4, T/2 or T - C) against the
    oracle restarted from the library's own state after s tokens."""
    w = WORKLOADS[name]
    inp, t, full = _full_call(name)
    s = {"quarter": w.T // 4, "half": w.T // 2, "last": w.T - w.C}[where]
    s -= s % w.C
    head = _run(w, t, T=s)
    units = _sample_units(w)
    tol = TOL[w.qkv_dtype]
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
        e = s + w.C
        y, W, S, _ = oracle.forward_unit(
            w, d["k"][s:e], d["q"][s:e], d["v"][s:e], d["theta"][s:e], d["eta"][s:e], d["alpha"][s:e],
            None if d["gamma"] is None else d["gamma"][s:e], W0, S0, d["P"], **kw)
        ey = maxrel(flat_units(full["y"])[u][s:e], y)
        msg = f"{name} unit {u} chunk at {s}: y {ey:.2e}"
        assert ey <= tol, msg
        if where == "last":
            eW = max(maxrel(flat_units(full["W"][m])[u], W[m]) for m in range(len(W)))
            eS = max(maxrel(flat_units(full["S"][m])[u], S[m]) for m in range(len(S)))
            msg += f"  W {eW:.2e}  S {eS:.2e}"
            assert eW <= tol and eS <= 5 * tol, msg
        print(msg)
