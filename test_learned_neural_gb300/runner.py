"""Tensor marshalling around the C entry points for whole workloads.

``Memory`` owns one library handle for a memory configuration; ``forward``
takes torch tensors (device or pinned host) in the layouts of
include/atlas_mem.h and returns the outputs.  No arithmetic of the method
happens here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (ATLAS_BF16, ATLAS_F32, atlas_mem_create, atlas_mem_destroy, atlas_mem_forward,
               atlas_mem_forward_host, atlas_mem_status, atlas_prologue_create, atlas_prologue_destroy,
               atlas_prologue_forward, atlas_prologue_io, atlas_prologue_last_gemm, atlas_prologue_status,
               current_stream, make_config, make_io, make_prologue_config, AtlasError)


def matrix_shapes(cfg):
    F = cfg.proj_dim if cfg.proj_dim else (cfg.d_k if cfg.p == 1 else (cfg.d_k + 1) * (cfg.d_k + 2) // 2)
    if cfg.depth == 1:
        return [(F, cfg.d_v)]
    return [(F, cfg.hidden), (cfg.hidden, cfg.d_v)]


class Memory:
    """A configured memory layer (one library handle)."""

    def __init__(self, cfg):
        self.cfg = cfg
        self.shapes = matrix_shapes(cfg)
        self.qkv_torch = torch.float32 if cfg.qkv_dtype in ("f32", ATLAS_F32) else torch.bfloat16
        self.h = atlas_mem_create(make_config(cfg.depth, cfg.d_k, cfg.d_v, cfg.hidden if cfg.depth == 2 else 0,
                                              cfg.C, cfg.c, cfg.p, cfg.proj_dim, cfg.ns_iters, cfg.qkv_dtype,
                                              getattr(cfg, "readout", "post"),
                                              getattr(cfg, "ns_target", "momentum"),
                                              getattr(cfg, "update", "per_token")))

    def close(self):
        if self.h is not None:
            atlas_mem_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc_outputs(self, B, H, T, device):
        f32 = torch.float32
        out = dict(
            y=torch.empty((B, H, T, self.cfg.d_v), dtype=f32, device=device),
            W=[torch.empty((B, H, r, c), dtype=f32, device=device) for r, c in self.shapes],
            S=[torch.empty((B, H, r, c), dtype=f32, device=device) for r, c in self.shapes],
        )
        nc = max(self.cfg.c - 1, 0)
        if nc:
            out["win_k"] = torch.zeros((B, H, nc, self.cfg.d_k), dtype=self.qkv_torch, device=device)
            out["win_v"] = torch.zeros((B, H, nc, self.cfg.d_v), dtype=self.qkv_torch, device=device)
            out["win_gamma"] = torch.zeros((B, H, nc), dtype=f32, device=device)
        return out

    def forward(self, t, out=None, win=None, host=False, stream=None):
        """t: dict of tensors (q, k, v, theta, eta, alpha, gamma, P, W0, S0);
        win: optional (win_len, win_k, win_v, win_gamma).  Returns the outputs."""
        B, H, T = t["q"].shape[:3]
        dev = "cpu" if host else t["q"].device
        if out is None:
            out = self.alloc_outputs(B, H, T, dev)
            if host:
                for key, val in list(out.items()):
                    out[key] = [x.pin_memory() for x in val] if isinstance(val, list) else val.pin_memory()
        win_len, wk, wv, wg = win if win is not None else (0, None, None, None)
        io = make_io(B, H, T, t["q"], t["k"], t["v"], t["theta"], t["eta"], t["alpha"], t.get("gamma"),
                     t.get("P"), t["W0"], t["S0"], out["y"], out["W"], out["S"],
                     win_len=win_len, win_k=wk, win_v=wv, win_gamma=wg,
                     win_k_out=out.get("win_k"), win_v_out=out.get("win_v"), win_gamma_out=out.get("win_gamma"))
        s = current_stream() if stream is None else stream
        if host:
            atlas_mem_forward_host(self.h, io, s)
        else:
            atlas_mem_forward(self.h, io, s)
        return out

    def status(self):
        rc = atlas_mem_status(self.h)
        if rc:
            raise AtlasError(rc, "device status")
        return rc


def tensors_from_numpy(inp: dict, device="cuda", pin=False):
    """Harness-style numpy inputs (bf16 as uint16 bit patterns) -> torch."""
    def conv(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(a)
        if device == "cpu":
            return t.pin_memory() if pin else t
        return t.to(device, non_blocking=False)

    out = {k: conv(inp[k]) for k in ("q", "k", "v", "theta", "eta", "alpha", "gamma", "P")}
    out["W0"] = [conv(m) for m in inp["W0"]]
    out["S0"] = [conv(m) for m in inp["S0"]]
    return out


class Prologue:
    """A configured stage in front of the memory (one library handle):
    x [B, T, D] -> q, k, v [B, H, T, d] and the gates [B, H, T]."""

    def __init__(self, cfg):
        self.cfg = cfg
        self.qkv_torch = torch.float32 if cfg.qkv_dtype in ("f32", ATLAS_F32) else torch.bfloat16
        self.h = atlas_prologue_create(make_prologue_config(cfg.D, cfg.H, cfg.d_k, cfg.d_v, cfg.conv,
                                                            cfg.with_gamma, cfg.theta_max, cfg.qkv_dtype))

    def close(self):
        if self.h is not None:
            atlas_prologue_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc_outputs(self, B, T, device):
        c, f32 = self.cfg, torch.float32
        out = dict(q=torch.empty((B, c.H, T, c.d_k), dtype=self.qkv_torch, device=device),
                   k=torch.empty((B, c.H, T, c.d_k), dtype=self.qkv_torch, device=device),
                   v=torch.empty((B, c.H, T, c.d_v), dtype=self.qkv_torch, device=device))
        for g in ("theta", "eta", "alpha") + (("gamma",) if c.with_gamma else ()):
            out[g] = torch.empty((B, c.H, T), dtype=f32, device=device)
        if c.conv > 1:
            out["cache"] = torch.empty((B, c.conv - 1, c.Nc), dtype=f32, device=device)
        return out

    def forward(self, t, out=None, stream=None):
        """t: dict of device tensors x, W_in, conv_w, gate_b and optional cache."""
        B, T = t["x"].shape[:2]
        if out is None:
            out = self.alloc_outputs(B, T, t["x"].device)

        def ptr(a):
            return None if a is None else a.data_ptr()

        io = atlas_prologue_io(B, T, ptr(t["x"]), ptr(t["W_in"]), ptr(t["conv_w"]), ptr(t["gate_b"]),
                               ptr(t.get("cache")), ptr(out["q"]), ptr(out["k"]), ptr(out["v"]), ptr(out["theta"]),
                               ptr(out["eta"]), ptr(out["alpha"]), ptr(out.get("gamma")), ptr(out.get("cache")))
        atlas_prologue_forward(self.h, io, current_stream() if stream is None else stream)
        return out

    def status(self):
        rc = atlas_prologue_status(self.h)
        if rc:
            raise AtlasError(rc, "device status of the stage in front of the memory")
        return rc

    def last_gemm(self):
        """1: the projection ran on the tensor cores (TMA + tcgen05), 0: fp32 SIMT."""
        return atlas_prologue_last_gemm(self.h)


def prologue_tensors_from_numpy(inp: dict, device="cuda"):
    """Seeded prologue inputs (bf16 as uint16 bit patterns) -> torch."""
    def conv(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)
    return {k: conv(inp.get(k)) for k in ("x", "W_in", "conv_w", "gate_b", "cache")}
