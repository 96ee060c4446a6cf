"""The depth-1 memory on polynomial features on the tensor cores (one
persistent launch per call, one cluster per unit): CUDA library vs the fp64
oracle over geometries that change the cluster size (the feature count F sets
how many CTAs share a unit's W, S), ragged chunk and value widths, both
read-out modes, the identity map, and calls chained through the carried
state and window cache (atlas-torch README, "Atlas Extensions": Polynomial
Features; ATLAS summary, Sec. 3.2: the Omega rule over a window of c keys).
"""
import numpy as np
import pytest

import oracle
from harness import WORKLOADS, make_inputs
from tests.gpu_common import TOL, compare, flat_units, maxrel, run_gpu

pytestmark = pytest.mark.gpu

BASE = WORKLOADS["atlas_poly_c4"]

CASES = [
    ("F561_c4", dict(B=1, H=2, T=256)),                       # 6 CTAs of 96 features
    ("F561_c16", dict(B=1, H=2, T=256, c=16)),                # 79 window rows
    ("F45", dict(B=2, H=1, T=192, d_k=8)),                    # one CTA of 48 features
    ("F153", dict(B=1, H=2, T=192, d_k=16)),                  # 2 CTAs of 80
    ("F325", dict(B=1, H=1, T=192, d_k=24)),                  # 4 CTAs of 96 (ragged last slice)
    ("C48_dv40", dict(B=1, H=2, T=192, C=48, d_v=40)),        # ragged rows and value columns
    ("C16_c1", dict(B=1, H=2, T=128, C=16, c=1)),             # short chunks, no window
    ("identity32", dict(B=1, H=2, T=192, p=1, d_k=32)),       # phi = identity, F = 32
]


def _launches(w):
    import test_learned_neural_gb300 as tln
    from test_learned_neural_gb300.runner import Memory, tensors_from_numpy
    mem = Memory(w)
    mem.forward(tensors_from_numpy(make_inputs(w)))
    mem.status()
    n = tln.atlas_mem_last_launches(mem.h)
    mem.close()
    return n


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("readout", ["post", "pre"])
def test_dual1_tc_parity(gpu_lib, name, kw, readout):
    w = BASE.scaled(**kw).scaled(readout=readout)
    # the persistent kernel ran (the split path takes three launches per chunk)
    assert _launches(w) <= 4
    errs = compare(w)
    tol = TOL[w.qkv_dtype]
    print(name, readout, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["y"] <= tol
    assert errs["W0"] <= tol and errs["S0"] <= 5 * tol


def test_dual1_tc_chained_calls_equal_one_call(gpu_lib):
    """Two calls, the second from the first's W, S and window cache, equal
    one call over the whole sequence bit for bit (the same kernel runs the
    same chunks from the same state)."""
    import torch
    from test_learned_neural_gb300.runner import Memory, tensors_from_numpy
    w = BASE.scaled(B=1, H=2, T=256, c=16)
    inp = make_inputs(w)
    whole = run_gpu(w, inp)
    t = tensors_from_numpy(inp)
    half = w.T // 2
    seq = ("q", "k", "v", "theta", "eta", "alpha", "gamma")
    first = {k: (v[:, :, :half].contiguous() if k in seq and v is not None else v) for k, v in t.items()}
    second = {k: (v[:, :, half:].contiguous() if k in seq and v is not None else v) for k, v in t.items()}
    mem = Memory(w)
    a = mem.forward(first)
    second["W0"], second["S0"] = a["W"], a["S"]
    b = mem.forward(second, win=(w.c - 1, a["win_k"], a["win_v"], a["win_gamma"]))
    torch.cuda.synchronize()
    mem.status()
    y = np.concatenate([a["y"].cpu().numpy(), b["y"].cpu().numpy()], axis=2)
    np.testing.assert_array_equal(y, whole["y"])
    np.testing.assert_array_equal(b["W"][0].cpu().numpy(), whole["W"][0])
    np.testing.assert_array_equal(b["S"][0].cpu().numpy(), whole["S"][0])
    mem.close()


def test_dual1_tc_full_size_prefix(gpu_lib):
    """Full-size atlas_poly_c16 in one call (the bench's launch): the first
    two chunks of two sampled units against the oracle from the true initial
    state; the later chunks (the memory passes fp32 range after about 17)
    still run and stay finite up to chunk 8."""
    w = WORKLOADS["atlas_poly_c16"]
    assert _launches(w) <= 4
    inp = make_inputs(w)
    g = run_gpu(w, inp)
    units = [0, w.units - 1]
    T0 = 2 * w.C
    r = oracle.forward(w, inp, units=units, T=T0)
    assert maxrel(flat_units(g["y"])[units][:, :T0], r["y"]) <= TOL[w.qkv_dtype]
    assert np.isfinite(flat_units(g["y"])[:, : 8 * w.C]).all()
