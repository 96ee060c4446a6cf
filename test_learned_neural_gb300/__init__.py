"""Python binding of the GB300 Titans/ATLAS memory-layer library.

The functions below carry the C entry points' names and only marshal
arguments (torch tensors -> device pointers, the current CUDA stream) into
``libatlas_mem.so``; every step of the forward runs in the library's CUDA
kernels.  There is no fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libatlas_mem.so")

ATLAS_OK, ATLAS_ERR_INVALID_ARG, ATLAS_ERR_UNSUPPORTED, ATLAS_ERR_CUDA, ATLAS_ERR_OOM, ATLAS_ERR_TIMEOUT, \
    ATLAS_ERR_RANGE = range(7)
ATLAS_F32, ATLAS_BF16 = 0, 1
ATLAS_READOUT_POST, ATLAS_READOUT_PRE = 0, 1
ATLAS_NS_MOMENTUM, ATLAS_NS_SURPRISE = 0, 1
ATLAS_UPDATE_PER_TOKEN, ATLAS_UPDATE_CHUNKWISE = 0, 1
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "OOM", 5: "TIMEOUT"}

# exported symbols, as declared in include/atlas_mem.h and include/atlas_prologue.h
EXPORTS = ("atlas_mem_create", "atlas_mem_forward", "atlas_mem_forward_host", "atlas_mem_forward_noalloc",
           "atlas_mem_status",
           "atlas_mem_workspace_bytes", "atlas_mem_last_launches", "atlas_mem_last_error", "atlas_mem_destroy",
           "atlas_prologue_create", "atlas_prologue_forward", "atlas_prologue_workspace_bytes",
           "atlas_prologue_last_error", "atlas_prologue_destroy", "atlas_prologue_status",
           "atlas_prologue_last_gemm")


class atlas_mem_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("depth", "d_k", "d_v", "hidden", "C", "c", "p", "proj_dim", "ns_iters", "qkv_dtype", "readout",
                                     "ns_target", "update")]


_vp = ctypes.c_void_p


class atlas_mem_io(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
        ("q", _vp), ("k", _vp), ("v", _vp),
        ("theta", _vp), ("eta", _vp), ("alpha", _vp), ("gamma", _vp),
        ("P", _vp),
        ("W0", _vp * 2), ("S0", _vp * 2),
        ("win_len", ctypes.c_int),
        ("win_k", _vp), ("win_v", _vp), ("win_gamma", _vp),
        ("y", _vp),
        ("W_out", _vp * 2), ("S_out", _vp * 2),
        ("win_k_out", _vp), ("win_v_out", _vp), ("win_gamma_out", _vp),
    ]


class atlas_prologue_config(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int), ("H", ctypes.c_int), ("d_k", ctypes.c_int), ("d_v", ctypes.c_int),
                ("conv", ctypes.c_int), ("with_gamma", ctypes.c_int), ("theta_max", ctypes.c_float),
                ("qkv_dtype", ctypes.c_int)]


class atlas_prologue_io(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int)] + [
        (n, _vp) for n in ("x", "W_in", "conv_w", "gate_b", "cache", "q", "k", "v", "theta", "eta", "alpha",
                           "gamma", "cache_out")]


class AtlasError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libatlas_mem.so is not built ({path}); run `python -m test_learned_neural_gb300.build`")
    lib = ctypes.CDLL(path)
    lib.atlas_mem_create.argtypes = [ctypes.POINTER(atlas_mem_config), ctypes.POINTER(ctypes.c_void_p)]
    lib.atlas_mem_create.restype = ctypes.c_int
    for name in ("atlas_mem_forward", "atlas_mem_forward_host", "atlas_mem_forward_noalloc"):
        fn = getattr(lib, name)
        fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(atlas_mem_io), ctypes.c_void_p]
        fn.restype = ctypes.c_int
    lib.atlas_mem_status.argtypes = [ctypes.c_void_p]
    lib.atlas_mem_status.restype = ctypes.c_int
    lib.atlas_mem_workspace_bytes.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.atlas_mem_workspace_bytes.restype = ctypes.c_size_t
    lib.atlas_mem_last_launches.argtypes = [ctypes.c_void_p]
    lib.atlas_mem_last_launches.restype = ctypes.c_int
    lib.atlas_mem_last_error.argtypes = [ctypes.c_void_p]
    lib.atlas_mem_last_error.restype = ctypes.c_char_p
    lib.atlas_mem_destroy.argtypes = [ctypes.c_void_p]
    lib.atlas_mem_destroy.restype = None
    lib.atlas_prologue_create.argtypes = [ctypes.POINTER(atlas_prologue_config), ctypes.POINTER(ctypes.c_void_p)]
    lib.atlas_prologue_create.restype = ctypes.c_int
    lib.atlas_prologue_forward.argtypes = [ctypes.c_void_p, ctypes.POINTER(atlas_prologue_io), ctypes.c_void_p]
    lib.atlas_prologue_forward.restype = ctypes.c_int
    lib.atlas_prologue_workspace_bytes.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    lib.atlas_prologue_workspace_bytes.restype = ctypes.c_size_t
    lib.atlas_prologue_last_error.argtypes = [ctypes.c_void_p]
    lib.atlas_prologue_last_error.restype = ctypes.c_char_p
    lib.atlas_prologue_destroy.argtypes = [ctypes.c_void_p]
    lib.atlas_prologue_destroy.restype = None
    lib.atlas_prologue_status.argtypes = [ctypes.c_void_p]
    lib.atlas_prologue_status.restype = ctypes.c_int
    lib.atlas_prologue_last_gemm.argtypes = [ctypes.c_void_p]
    lib.atlas_prologue_last_gemm.restype = ctypes.c_int
    _lib = lib
    return lib


# ------------------------------------------------------------ C entry points
def atlas_mem_create(cfg: atlas_mem_config):
    lib = load()
    h = ctypes.c_void_p()
    rc = lib.atlas_mem_create(ctypes.byref(cfg), ctypes.byref(h))
    if rc:
        raise AtlasError(rc, lib.atlas_mem_last_error(None).decode())
    return h


def atlas_mem_forward(h, io: atlas_mem_io, stream: int = 0):
    lib = load()
    rc = lib.atlas_mem_forward(h, ctypes.byref(io), ctypes.c_void_p(stream))
    if rc:
        raise AtlasError(rc, lib.atlas_mem_last_error(h).decode())


def atlas_mem_forward_host(h, io: atlas_mem_io, stream: int = 0):
    lib = load()
    rc = lib.atlas_mem_forward_host(h, ctypes.byref(io), ctypes.c_void_p(stream))
    if rc:
        raise AtlasError(rc, lib.atlas_mem_last_error(h).decode())


def atlas_mem_forward_noalloc(h, io: atlas_mem_io, stream: int = 0):
    """atlas_mem_forward without any device allocation (fixed scratch)."""
    lib = load()
    rc = lib.atlas_mem_forward_noalloc(h, ctypes.byref(io), ctypes.c_void_p(stream))
    if rc:
        raise AtlasError(rc, lib.atlas_mem_last_error(h).decode())


def atlas_mem_status(h) -> int:
    return load().atlas_mem_status(h)


def atlas_mem_workspace_bytes(h, B, H, T) -> int:
    return load().atlas_mem_workspace_bytes(h, B, H, T)


def atlas_mem_last_launches(h) -> int:
    return load().atlas_mem_last_launches(h)


def atlas_mem_last_error(h) -> str:
    return load().atlas_mem_last_error(h).decode()


def atlas_prologue_create(cfg: atlas_prologue_config):
    lib = load()
    h = ctypes.c_void_p()
    rc = lib.atlas_prologue_create(ctypes.byref(cfg), ctypes.byref(h))
    if rc:
        raise AtlasError(rc, lib.atlas_prologue_last_error(None).decode())
    return h


def atlas_prologue_forward(h, io: atlas_prologue_io, stream: int = 0):
    lib = load()
    rc = lib.atlas_prologue_forward(h, ctypes.byref(io), ctypes.c_void_p(stream))
    if rc:
        raise AtlasError(rc, lib.atlas_prologue_last_error(h).decode())


def atlas_prologue_workspace_bytes(h, B, T) -> int:
    return load().atlas_prologue_workspace_bytes(h, B, T)


def atlas_prologue_last_error(h) -> str:
    return load().atlas_prologue_last_error(h).decode()


def atlas_prologue_status(h) -> int:
    return load().atlas_prologue_status(h)


def atlas_prologue_last_gemm(h) -> int:
    return load().atlas_prologue_last_gemm(h)


def atlas_prologue_destroy(h):
    load().atlas_prologue_destroy(h)


def make_prologue_config(D, H, d_k, d_v, conv, with_gamma, theta_max, qkv_dtype) -> atlas_prologue_config:
    dt = {"f32": ATLAS_F32, "bf16": ATLAS_BF16}.get(qkv_dtype, qkv_dtype)
    return atlas_prologue_config(D, H, d_k, d_v, conv, int(with_gamma), theta_max, dt)


def atlas_mem_destroy(h):
    load().atlas_mem_destroy(h)


# ------------------------------------------------------------- marshalling
def make_config(depth, d_k, d_v, hidden, C, c, p, proj_dim, ns_iters, qkv_dtype,
                readout="post", ns_target="momentum", update="per_token") -> atlas_mem_config:
    dt = {"f32": ATLAS_F32, "bf16": ATLAS_BF16}.get(qkv_dtype, qkv_dtype)
    ro = {"post": ATLAS_READOUT_POST, "pre": ATLAS_READOUT_PRE}.get(readout, readout)
    nt = {"momentum": ATLAS_NS_MOMENTUM, "surprise": ATLAS_NS_SURPRISE}.get(ns_target, ns_target)
    up = {"per_token": ATLAS_UPDATE_PER_TOKEN, "chunkwise": ATLAS_UPDATE_CHUNKWISE}.get(update, update)
    return atlas_mem_config(depth, d_k, d_v, hidden, C, c, p, proj_dim, ns_iters, dt, ro, nt, up)


def _ptr(t):
    return None if t is None else t.data_ptr()


def make_io(B, H, T, q, k, v, theta, eta, alpha, gamma, P, W0, S0, y, W_out, S_out,
            win_len=0, win_k=None, win_v=None, win_gamma=None,
            win_k_out=None, win_v_out=None, win_gamma_out=None) -> atlas_mem_io:
    """Pack tensors (torch, device or host) into the C struct.  Tensors must be
    contiguous with the layouts given in include/atlas_mem.h; W0/S0/W_out/S_out
    are lists of one tensor per memory matrix."""
    io = atlas_mem_io()
    io.B, io.H, io.T = B, H, T
    io.q, io.k, io.v = _ptr(q), _ptr(k), _ptr(v)
    io.theta, io.eta, io.alpha, io.gamma = _ptr(theta), _ptr(eta), _ptr(alpha), _ptr(gamma)
    io.P = _ptr(P)
    for m in range(2):
        io.W0[m] = _ptr(W0[m]) if m < len(W0) else None
        io.S0[m] = _ptr(S0[m]) if m < len(S0) else None
        io.W_out[m] = _ptr(W_out[m]) if m < len(W_out) else None
        io.S_out[m] = _ptr(S_out[m]) if m < len(S_out) else None
    io.win_len = win_len
    io.win_k, io.win_v, io.win_gamma = _ptr(win_k), _ptr(win_v), _ptr(win_gamma)
    io.y = _ptr(y)
    io.win_k_out, io.win_v_out, io.win_gamma_out = _ptr(win_k_out), _ptr(win_v_out), _ptr(win_gamma_out)
    for t in (q, k, v, theta, eta, alpha, gamma, P, y, win_k, win_v, win_gamma,
              win_k_out, win_v_out, win_gamma_out, *W0, *S0, *W_out, *S_out):
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    return io


def current_stream() -> int:
    import torch
    return torch.cuda.current_stream().cuda_stream
