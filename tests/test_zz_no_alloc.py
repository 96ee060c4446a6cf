"""atlas_mem_forward_noalloc: the forward for callers that must not allocate
device memory (a host framework whose pool owns the GPU's memory, or a
serving loop that forbids cudaMalloc after start-up).  It works in a fixed
device array inside the library instead of a workspace it allocates.

Its output must match atlas_mem_forward's on the same inputs, on calls made
back to back (the fixed array keeps the previous call's contents), and calls
too large for the array must be refused with a clear message.  This file is
collected last on purpose: if it fails, every other test has already run.
"""
import ctypes

import numpy as np
import pytest

import test_learned_neural_gb300 as tln
from harness import WORKLOADS, make_inputs
from tests.gpu_common import TOL, maxrel


def _call(entry, w, inp):
    import torch
    from test_learned_neural_gb300.runner import Memory, tensors_from_numpy
    mem = Memory(w)
    t = tensors_from_numpy(inp, device="cuda")
    out = mem.alloc_outputs(w.B, w.H, w.T, "cuda")
    io = tln.make_io(w.B, w.H, w.T, t["q"], t["k"], t["v"], t["theta"], t["eta"], t["alpha"], t["gamma"], t["P"],
                     t["W0"], t["S0"], out["y"], out["W"], out["S"], win_k_out=out.get("win_k"),
                     win_v_out=out.get("win_v"), win_gamma_out=out.get("win_gamma"))
    entry(mem.h, io, tln.current_stream())
    torch.cuda.synchronize()
    assert tln.atlas_mem_status(mem.h) == tln.ATLAS_OK
    res = [out["y"].cpu().numpy()] + [m.cpu().numpy() for m in out["W"] + out["S"]]
    mem.close()
    return res


@pytest.mark.gpu
def test_noalloc_matches_forward_on_calls_in_a_row(gpu_lib):
    cases = [WORKLOADS["titans_mlp"].scaled(B=1, H=2, T=256),
             WORKLOADS["atlas_long"].scaled(B=1, H=1, T=128)]
    for w in cases:
        h = tln.atlas_mem_create(tln.make_config(w.depth, w.d_k, w.d_v, w.hidden, w.C, w.c, w.p, w.proj_dim,
                                                 w.ns_iters, w.qkv_dtype))
        assert tln.atlas_mem_workspace_bytes(h, w.B, w.H, w.T) <= 16 * 1024 * 1024
        tln.atlas_mem_destroy(h)
    inps = [make_inputs(w) for w in cases]
    refs = [_call(tln.atlas_mem_forward, w, i) for w, i in zip(cases, inps)]
    # back to back: A, B, then A again over B's leftovers in the fixed array
    gots = []
    for w, inp, ref in [(cases[0], inps[0], refs[0]), (cases[1], inps[1], refs[1]), (cases[0], inps[0], refs[0])]:
        got = _call(tln.atlas_mem_forward_noalloc, w, inp)
        gots.append(got)
        tol = TOL[w.qkv_dtype]
        for g, r in zip(got, ref):
            assert maxrel(g, r) <= tol
    # the same kernels on the same inputs: any difference between the first
    # and the third call could only come from B's leftovers in the array
    for a, b in zip(gots[0], gots[2]):
        assert np.array_equal(a, b)
    # and the same kernels as atlas_mem_forward: equal bit for bit
    for g, r in zip(gots[0], refs[0]):
        assert np.array_equal(g, r)
    for g, r in zip(gots[1], refs[1]):
        assert np.array_equal(g, r)


@pytest.mark.gpu
def test_noalloc_runs_the_fused_kernel_at_full_size(gpu_lib):
    """The fused MLP kernel needs only the array's status word: the full
    Titans workload, far beyond the array, runs and equals atlas_mem_forward."""
    w = WORKLOADS["titans_mlp"]
    inp = make_inputs(w)
    ref = _call(tln.atlas_mem_forward, w, inp)
    got = _call(tln.atlas_mem_forward_noalloc, w, inp)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_noalloc_refuses_calls_beyond_its_scratch():
    """Refused on the host before any CUDA call (runs without a GPU)."""
    import os
    from test_learned_neural_gb300 import build as tln_build
    if not os.path.exists(tln.LIB_PATH):
        tln_build.build()
    lib = tln.load()
    w = WORKLOADS["atlas_muon"]          # full size: far beyond 16 MiB of scratch (multi-launch path)
    h = tln.atlas_mem_create(tln.make_config(w.depth, w.d_k, w.d_v, w.hidden, w.C, w.c, w.p, w.proj_dim,
                                             w.ns_iters, w.qkv_dtype))
    try:
        need = tln.atlas_mem_workspace_bytes(h, w.B, w.H, w.T)
        assert need > 16 * 1024 * 1024
        dummy = np.zeros(16, np.float32)   # never dereferenced: the size check comes first
        p = dummy.ctypes.data
        io = tln.atlas_mem_io()
        io.B, io.H, io.T = w.B, w.H, w.T
        for f in ("q", "k", "v", "theta", "eta", "alpha", "y"):
            setattr(io, f, p)
        for m in range(2):
            io.W0[m] = io.S0[m] = io.W_out[m] = io.S_out[m] = p
        rc = lib.atlas_mem_forward_noalloc(h, ctypes.byref(io), None)
        assert rc == tln.ATLAS_ERR_UNSUPPORTED
        msg = tln.atlas_mem_last_error(h)
        assert str(need) in msg and str(16 * 1024 * 1024) in msg
    finally:
        tln.atlas_mem_destroy(h)
