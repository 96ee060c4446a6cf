"""Seeded synthetic inputs for the memory-layer forward.

Recipe (one ``numpy.random.default_rng(seed)`` per workload, draws in this
order): k, q, v, theta, eta, alpha, gamma (only where the workload uses
per-token Omega weights), W0 (only for Xavier-initialised memories), P (only
where features are projected).

* k, q ~ N(0, 1), L2-normalised per token, then stored in the input precision
  (float32, or bf16 by round-to-nearest-even).
* v ~ N(0, 1), same storage.
* theta = theta_scale * sigmoid(N(0, 1)) (theta_scale 0.1, or 0.1 / C on the
  chunk-wise Titans workload, whose chunk sums C gradients), eta = sigmoid(N(1, 1)),
  alpha = sigmoid(N(alpha_mu, 1)), gamma = sigmoid(N(0, 1)); all float32.
* W0: zeros, or Xavier-normal (std sqrt(2 / (fan_in + fan_out))) drawn once per
  head and shared by every batch row; S0 = 0.  float32.
* P ~ N(0, 1 / F) with F the monomial count, rounded to bf16.

Layouts: q, k, v are [B, H, T, d] row-major; gates [B, H, T]; each weight
matrix [B, H, rows, cols]; P [F, proj_dim].  bf16 arrays are returned as their
uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np

from .configs import Workload


def bf16_bits(x) -> np.ndarray:
    """float -> bf16 bit pattern (uint16), round to nearest, ties to even."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_from_bits(b) -> np.ndarray:
    """bf16 bit pattern (uint16) -> exact float32 values."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_round(x) -> np.ndarray:
    """Round to the nearest bf16 value, returned as float32."""
    return bf16_from_bits(bf16_bits(x))


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def _l2n(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _store(x, dtype):
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits(x)
    raise ValueError(dtype)


def make_inputs(w: Workload) -> dict:
    rng = np.random.default_rng(w.seed)
    B, H, T = w.B, w.H, w.T
    out = {}
    out["k"] = _store(_l2n(rng.standard_normal((B, H, T, w.d_k))), w.qkv_dtype)
    out["q"] = _store(_l2n(rng.standard_normal((B, H, T, w.d_k))), w.qkv_dtype)
    out["v"] = _store(rng.standard_normal((B, H, T, w.d_v)), w.qkv_dtype)
    f32 = np.float32
    out["theta"] = (w.theta_scale * _sigmoid(rng.standard_normal((B, H, T)))).astype(f32)
    out["eta"] = _sigmoid(rng.normal(1.0, 1.0, (B, H, T))).astype(f32)
    out["alpha"] = _sigmoid(rng.normal(w.alpha_mu, 1.0, (B, H, T))).astype(f32)
    out["gamma"] = (_sigmoid(rng.standard_normal((B, H, T))).astype(f32)
                    if w.use_gamma else None)
    W0 = []
    for (r, c) in w.matrix_shapes():
        if w.w0_init == "xavier":
            per_head = rng.normal(0.0, np.sqrt(2.0 / (r + c)), (H, r, c))
            W0.append(np.ascontiguousarray(
                np.broadcast_to(per_head[None], (B, H, r, c)), dtype=f32))
        else:
            W0.append(np.zeros((B, H, r, c), f32))
    out["W0"] = W0
    out["S0"] = [np.zeros_like(m) for m in W0]
    if w.proj_dim:
        F = w.poly_dim
        out["P"] = bf16_bits(rng.normal(0.0, np.sqrt(1.0 / F), (F, w.proj_dim)))
    else:
        out["P"] = None
    return out


def unit_slice(inp: dict, w: Workload, units) -> dict:
    """Restrict inputs to a list of flattened (b*H + h) unit indices.

    The result has shape B=len(units), H=1 in every per-unit array."""
    units = list(units)
    sel = {}
    for key in ("k", "q", "v", "theta", "eta", "alpha", "gamma"):
        a = inp[key]
        if a is None:
            sel[key] = None
            continue
        flat = a.reshape((w.B * w.H,) + a.shape[2:])
        sel[key] = np.ascontiguousarray(flat[units][:, None])
    for key in ("W0", "S0"):
        sel[key] = [np.ascontiguousarray(m.reshape((w.B * w.H,) + m.shape[2:])[units][:, None])
                    for m in inp[key]]
    sel["P"] = inp["P"]
    return sel


def make_prologue_inputs(p, cache=False) -> dict:
    """Seeded inputs of the stage in front of the memory.

    One ``default_rng(seed)``, drawing in order: x ~ N(0, 1) [B, T, D];
    W_in ~ N(0, 1 / D) [D, N]; conv taps ~ N(0, 1 / conv) [Nc, conv]; gate
    biases (theta 0, eta 1, alpha ``alpha_bias``, gamma 0, the centres of the
    memory inputs' gate draws) plus N(0, 0.1) per head [G, H]; with
    ``cache``, a carried convolution cache ~ N(0, 1) [B, conv - 1, Nc].
    x and W_in are stored in ``qkv_dtype``; the rest is float32."""
    rng = np.random.default_rng(p.seed)
    f32 = np.float32
    out = {}
    out["x"] = _store(rng.standard_normal((p.B, p.T, p.D)), p.qkv_dtype)
    out["W_in"] = _store(rng.normal(0.0, np.sqrt(1.0 / p.D), (p.D, p.N)), p.qkv_dtype)
    out["conv_w"] = rng.normal(0.0, np.sqrt(1.0 / p.conv), (p.Nc, p.conv)).astype(f32)
    centres = np.array([0.0, 1.0, p.alpha_bias, 0.0][:p.G])
    out["gate_b"] = (centres[:, None] + rng.normal(0.0, 0.1, (p.G, p.H))).astype(f32)
    out["cache"] = (rng.standard_normal((p.B, p.conv - 1, p.Nc)).astype(f32) if cache else None)
    return out
