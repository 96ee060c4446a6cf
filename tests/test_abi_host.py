"""Host-only checks of the C ABI: the library builds and loads, exports every
entry point the header declares, and rejects bad configs and calls before
touching the GPU."""
import ctypes
import os
import re

import pytest

import test_learned_neural_gb300 as tln
from test_learned_neural_gb300 import build as tln_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(tln.LIB_PATH):
        tln_build.build()
    return tln.load()


def declared_entry_points():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(atlas_\w+)\s*\(", src, re.M))
    return names


def test_header_declares_the_entry_points():
    assert set(tln.EXPORTS) <= declared_entry_points()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), name


def _cfg(**kw):
    base = dict(depth=2, d_k=64, d_v=64, hidden=256, C=64, c=1, p=1, proj_dim=0, ns_iters=0, qkv_dtype="bf16")
    base.update(kw)
    return tln.make_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(depth=3), tln.ATLAS_ERR_INVALID_ARG),
    (dict(d_v=32), tln.ATLAS_ERR_INVALID_ARG),            # residual needs F == d_v
    (dict(C=0), tln.ATLAS_ERR_INVALID_ARG),
    (dict(c=0), tln.ATLAS_ERR_INVALID_ARG),
    (dict(p=3), tln.ATLAS_ERR_INVALID_ARG),
    (dict(qkv_dtype=7), tln.ATLAS_ERR_INVALID_ARG),
    (dict(readout=5), tln.ATLAS_ERR_INVALID_ARG),
    (dict(C=2048), tln.ATLAS_ERR_UNSUPPORTED),            # window rows > 1024
    (dict(ns_target=3), tln.ATLAS_ERR_INVALID_ARG),
    (dict(ns_target=1, ns_iters=5, c=40), tln.ATLAS_ERR_INVALID_ARG),
    (dict(C=1000, c=100), tln.ATLAS_ERR_UNSUPPORTED),     # window rows > 1024
    (dict(update=2), tln.ATLAS_ERR_INVALID_ARG),
    (dict(update="chunkwise", c=2), tln.ATLAS_ERR_INVALID_ARG),           # no Omega window on that path
    (dict(update="chunkwise", ns_iters=5, ns_target="surprise"), tln.ATLAS_ERR_INVALID_ARG),
    (dict(d_k=256, d_v=256, hidden=512, ns_iters=5), tln.ATLAS_ERR_UNSUPPORTED),  # NS short side > 128
])
def test_create_rejects(lib, kw, code):
    with pytest.raises(tln.AtlasError) as ei:
        tln.atlas_mem_create(_cfg(**kw))
    assert ei.value.code == code
    assert tln.atlas_mem_last_error(None)


def test_create_accepts_every_named_workload(lib):
    from harness import WORKLOADS
    for w in WORKLOADS.values():
        h = tln.atlas_mem_create(tln.make_config(w.depth, w.d_k, w.d_v, w.hidden, w.C, w.c, w.p, w.proj_dim,
                                                 w.ns_iters, w.qkv_dtype, w.readout, w.ns_target, w.update))
        assert tln.atlas_mem_workspace_bytes(h, w.B, w.H, w.T) > 0
        tln.atlas_mem_destroy(h)


def test_forward_validates_before_any_cuda_call(lib):
    h = tln.atlas_mem_create(_cfg())
    try:
        rc = lib.atlas_mem_forward(h, None, None)
        assert rc == tln.ATLAS_ERR_INVALID_ARG
        io = tln.atlas_mem_io()
        io.B, io.H, io.T = 1, 1, 100          # not a multiple of C = 64
        assert lib.atlas_mem_forward(h, ctypes.byref(io), None) == tln.ATLAS_ERR_UNSUPPORTED
        io.T = 128                            # now null tensors
        assert lib.atlas_mem_forward(h, ctypes.byref(io), None) == tln.ATLAS_ERR_INVALID_ARG
        assert "non-NULL" in tln.atlas_mem_last_error(h)
        io.B = 0
        assert lib.atlas_mem_forward_host(h, ctypes.byref(io), None) == tln.ATLAS_ERR_INVALID_ARG
    finally:
        tln.atlas_mem_destroy(h)


def test_null_handle(lib):
    assert lib.atlas_mem_forward(None, None, None) == tln.ATLAS_ERR_INVALID_ARG
    assert lib.atlas_mem_status(None) == tln.ATLAS_ERR_INVALID_ARG
    lib.atlas_mem_destroy(None)


def _pcfg(**kw):
    base = dict(D=32, H=2, d_k=8, d_v=8, conv=4, with_gamma=1, theta_max=0.1, qkv_dtype="bf16")
    base.update(kw)
    return tln.make_prologue_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(D=0), tln.ATLAS_ERR_INVALID_ARG),
    (dict(H=0), tln.ATLAS_ERR_INVALID_ARG),
    (dict(conv=0), tln.ATLAS_ERR_INVALID_ARG),
    (dict(with_gamma=2), tln.ATLAS_ERR_INVALID_ARG),
    (dict(theta_max=0.0), tln.ATLAS_ERR_INVALID_ARG),
    (dict(theta_max=float("inf")), tln.ATLAS_ERR_INVALID_ARG),
    (dict(qkv_dtype=7), tln.ATLAS_ERR_INVALID_ARG),
    (dict(conv=9), tln.ATLAS_ERR_UNSUPPORTED),
    (dict(d_k=200, d_v=200), tln.ATLAS_ERR_UNSUPPORTED),  # 2 d_k + d_v > 512 per head
])
def test_prologue_create_rejects(lib, kw, code):
    with pytest.raises(tln.AtlasError) as ei:
        tln.atlas_prologue_create(_pcfg(**kw))
    assert ei.value.code == code
    assert tln.atlas_prologue_last_error(None)


def test_prologue_forward_validates_before_any_cuda_call(lib):
    import ctypes
    h = tln.atlas_prologue_create(_pcfg())
    try:
        assert lib.atlas_prologue_forward(h, None, None) == tln.ATLAS_ERR_INVALID_ARG
        io = tln.atlas_prologue_io()
        io.B, io.T = 1, 0
        assert lib.atlas_prologue_forward(h, ctypes.byref(io), None) == tln.ATLAS_ERR_INVALID_ARG
        io.T = 16                              # null tensors
        assert lib.atlas_prologue_forward(h, ctypes.byref(io), None) == tln.ATLAS_ERR_INVALID_ARG
        assert "non-NULL" in tln.atlas_prologue_last_error(h)
        for name in ("x", "W_in", "conv_w", "gate_b", "q", "k", "v", "theta", "eta", "alpha"):
            setattr(io, name, 16)              # never dereferenced: validation fails first
        assert lib.atlas_prologue_forward(h, ctypes.byref(io), None) == tln.ATLAS_ERR_INVALID_ARG
        assert "gamma" in tln.atlas_prologue_last_error(h)
        io.gamma = 16
        io.cache = io.cache_out = 32
        assert lib.atlas_prologue_forward(h, ctypes.byref(io), None) == tln.ATLAS_ERR_INVALID_ARG
        assert "alias" in tln.atlas_prologue_last_error(h)
        # the fp32 projection (rounded to 256 bytes), W_in transposed for the
        # tensor-core GEMM (bf16 [N][D]: 56 x 32), 256 bytes for the status word
        N = 2 * (2 * 8 + 8) + 4 * 2
        assert tln.atlas_prologue_workspace_bytes(h, 2, 16) == -(-2 * 16 * N * 4 // 256) * 256 + N * 32 * 2 + 256
    finally:
        tln.atlas_prologue_destroy(h)
    lib.atlas_prologue_destroy(None)
