"""Helpers shared by the GPU parity tests (oracle vs CUDA library)."""
import numpy as np

import oracle
from harness import make_inputs

# Tolerances on max|gpu - ref| / max|ref| per output tensor: fp32 inputs 1e-4,
# bf16 inputs with fp32 accumulation 2e-2 (y and the final W).
TOL = {"f32": 1e-4, "bf16": 2e-2}


def maxrel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / (den if den > 0 else 1.0))


def run_gpu(w, inp, win=None, host=False):
    import torch
    from test_learned_neural_gb300.runner import Memory, tensors_from_numpy
    mem = Memory(w)
    t = tensors_from_numpy(inp, device="cpu" if host else "cuda", pin=host)
    out = mem.forward(t, win=win, host=host)
    if not host:
        torch.cuda.synchronize()
    mem.status()
    res = dict(y=out["y"].cpu().numpy(), W=[m.cpu().numpy() for m in out["W"]],
               S=[m.cpu().numpy() for m in out["S"]])
    for key in ("win_k", "win_v", "win_gamma"):
        if key in out:
            res[key] = out[key].cpu()
    mem.close()
    return res


def flat_units(a):
    a = np.asarray(a)
    return a.reshape((-1,) + a.shape[2:])


def compare(w, units=None, T=None):
    """Run GPU and oracle on workload w; return dict of max-rel errors."""
    inp = make_inputs(w)
    g = run_gpu(w, inp)
    r = oracle.forward(w, inp, units=units, T=T)
    sel = slice(None) if units is None else list(units)
    gy = flat_units(g["y"])[sel]
    if T is not None:
        gy = gy[:, :T]
    errs = {"y": maxrel(gy, r["y"])}
    if T is None:
        for m in range(len(r["W"])):
            errs[f"W{m}"] = maxrel(flat_units(g["W"][m])[sel], r["W"][m])
            errs[f"S{m}"] = maxrel(flat_units(g["S"][m])[sel], r["S"][m])
    return errs
