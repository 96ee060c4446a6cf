"""Plain fp64 oracle of the chunked Titans/ATLAS memory-layer forward.

TEST INFRASTRUCTURE ONLY: used by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; never by the library.  It shares no code
with the CUDA path.

Every (batch, head) unit is independent.  Per unit, token by token, in the
order the pages define:

* features   x_i = phi(k_i), r_t = phi(q_t); phi is the identity (p = 1) or the
             exact degree-2 monomial expansion [1, x_i, x_i x_j / 2 (i <= j)]
             with 1/m! on every degree-m monomial, optionally times P
             (atlas-torch README, "Atlas Extensions": Polynomial Features;
             ATLAS summary, Section 3.1).
* memory     M_W(x) = x W (depth 1) or x + SiLU(x W1) W2 (depth 2), row
             vectors, no biases (titans-pytorch-mlx README, "Key Innovations"
             3; ATLAS summary, Section 5.1: residual two-layer MLP).
* loss       l_i(W) = ||M_W(x_i) - v_i||^2, a plain sum of squares
             (titans-pytorch-mlx README, Eq. 12).
* chunks     tokens are cut into chunks of C; inside a chunk every gradient is
             taken at the chunk-start weights W_bar (ATLAS summary, Sections
             3.3 and 5.1; atlas-torch README, "Bug Fixes": per-token store path
             with gradients at segment-start weights).
* Omega      g_t = sum_{i = max(t0, t-c+1)}^{t} gamma_i grad l_i(W_bar): the last
             c tokens including t, crossing chunk edges, truncated at the start
             of the call unless earlier tokens are handed in as a window cache
             (ATLAS summary, Section 3.2; atlas-torch README, "Atlas
             Extensions": Omega Rule, and "Bug Fixes": Omega window slide).
* momentum   S_t = eta_t S_{t-1} - theta_t g_t (titans-pytorch-mlx README,
             Eq. 14).
* Muon       U_t = NS_k(S_t) per weight matrix when k > 0, else U_t = S_t; the
             raw S_t is what recurs (ATLAS summary, Section 5; atlas-torch
             README, "Atlas Extensions": Muon / Newton-Schulz).
* decay      W_t = (1 - alpha_t) W_{t-1} + U_t (titans-pytorch-mlx README,
             Eq. 13).
* read-out   y_t = M_{W_t}(r_t) from the post-update state of token t
             (atlas-torch README, "Known deviations from the paper's MAC").

The chunk-wise update rule (``update = "chunkwise"``) is the titans-pytorch
store path that the atlas-torch README sets beside the per-token one ("Bug
Fixes": the per_token_updates flag): one gradient per chunk, summed over its
tokens at W_bar, the chunk's momentum and decay gates pooled, one momentum /
decay step per chunk, and a read-out per chunk.
"""
from __future__ import annotations

import numpy as np

from harness.inputs import bf16_from_bits

# Muon quintic Newton-Schulz coefficients (a, b, c) and the normalisation eps.
NS_COEFFS = (3.4445, -4.7750, 2.0315)
NS_EPS = 1e-7


# ----------------------------------------------------------------- features
def poly_features(x: np.ndarray, p: int) -> np.ndarray:
    """Exact monomial expansion of degree <= p (p in {1, 2}).

    p = 1 returns x unchanged.  p = 2 returns [1, x_0..x_{d-1}, x_i x_j / 2!]
    over pairs i <= j in lexicographic (combinations-with-replacement) order,
    so the width is 1 + d + d(d+1)/2 (atlas-torch README, "Atlas Extensions":
    Polynomial Features; ATLAS summary, Section 3.1)."""
    x = np.asarray(x, dtype=np.float64)
    if p == 1:
        return x
    if p != 2:
        raise ValueError("only degrees 1 and 2 are defined here")
    d = x.shape[-1]
    iu, ju = np.triu_indices(d)
    const = np.ones(x.shape[:-1] + (1,))
    quad = 0.5 * x[..., iu] * x[..., ju]
    return np.concatenate([const, x, quad], axis=-1)


def features(x: np.ndarray, p: int, P=None) -> np.ndarray:
    """phi(x), optionally projected back by P (rows = monomials)."""
    f = poly_features(x, p)
    if P is not None:
        f = f @ np.asarray(P, dtype=np.float64)
    return f


# ------------------------------------------------------------------- memory
def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * _sigmoid(z)


def dsilu(z):
    s = _sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def memory_apply(W, x, depth):
    """M_W(x) for row vectors x [n, F]."""
    if depth == 1:
        return x @ W[0]
    return x + silu(x @ W[0]) @ W[1]


def token_gradients(W, X, V, depth):
    """Per-token gradients of l_i(W) = ||M_W(x_i) - v_i||^2.

    Returns one array [n, rows, cols] per weight matrix.  Depth 1 gives the
    delta-rule outer product 2 x_i^T (x_i W - v_i) (atlas-torch README, "How the
    memory works"); depth 2 is the chain rule through the residual SiLU MLP."""
    if depth == 1:
        dY = 2.0 * (X @ W[0] - V)
        return [np.einsum("ni,nj->nij", X, dY)]
    Z = X @ W[0]
    A = silu(Z)
    dY = 2.0 * (X + A @ W[1] - V)
    dZ = (dY @ W[1].T) * dsilu(Z)
    return [np.einsum("ni,nj->nij", X, dZ), np.einsum("ni,nj->nij", A, dY)]


def newton_schulz(G, steps, coeffs=NS_COEFFS, eps=NS_EPS):
    """Muon's quintic Newton-Schulz orthogonalisation, `steps` iterations.

    Works on the short side (transposes when rows > cols), normalises by the
    Frobenius norm plus eps, then repeats X <- a X + (b A + c A^2) X with
    A = X X^T (atlas-torch README, "Atlas Extensions": Muon / Newton-Schulz;
    ATLAS summary, Section 5)."""
    a, b, c = coeffs
    G = np.asarray(G, dtype=np.float64)
    tall = G.shape[0] > G.shape[1]
    X = G.T if tall else G
    X = X / (np.linalg.norm(X) + eps)
    for _ in range(steps):
        A = X @ X.T
        Bm = b * A + c * (A @ A)
        X = a * X + Bm @ X
    return X.T if tall else X


# ------------------------------------------------------------------ forward
def forward_unit(cfg, k, q, v, theta, eta, alpha, gamma, W0, S0, P=None,
                 cache_k=None, cache_v=None, cache_g=None):
    """Forward of one (batch, head) unit.

    k, q [T, d_k]; v [T, d_v]; theta, eta, alpha, gamma [T] (gamma None = 1);
    W0, S0 lists of matrices; cache_* hold up to c-1 tokens that precede this
    call (raw keys, values, Omega weights; oldest first).

    Returns y [T, d_v], W_T, S_T (lists) and the outgoing cache
    (the last min(c-1, cached + T) raw keys, values and weights)."""
    depth, C, c = cfg.depth, cfg.C, cfg.c
    # Read-out: "post" (default) reads token t with the memory after its own
    # update, as the atlas-torch implementation does (atlas-torch README,
    # "Known deviations from the paper's MAC"); "pre" reads it with the
    # memory before the update, h_t = M*_{t-1}(q_t) (titans-pytorch-mlx
    # README, MAC, Eq. 21).  The state itself is the same in both modes.
    pre = getattr(cfg, "readout", "post") == "pre"
    # Where Newton-Schulz sits (with ns_iters > 0): "momentum" (default)
    # orthogonalises the applied momentum, U_t = NS(S_t) (ATLAS summary,
    # Section 5); "surprise" orthogonalises each token's windowed gradient
    # with the momentum and step size outside it, S_t = eta_t S_{t-1} -
    # theta_t NS(g_t), W_t = (1 - alpha_t) W_{t-1} + S_t (atlas-torch README:
    # "orthogonalization of the surprise updates", per-token store path with
    # "eta outside Newton-Schulz").
    surprise_ns = bool(cfg.ns_iters) and getattr(cfg, "ns_target", "momentum") == "surprise"
    # Update rule: "per_token" (default, everything above) or "chunkwise", the
    # titans-pytorch chunk-wise store path (atlas-torch README, "Bug Fixes":
    # per_token_updates): per chunk, G = sum_i theta_i gamma_i grad l_i(W_bar)
    # over its tokens, the gates eta and alpha pooled to their mean over the
    # chunk, S <- eta_bar S - G, U = NS_k(S) (eta inside Newton-Schulz) or S,
    # W <- (1 - alpha_bar) W + U.  The memory exists only at chunk ends: token
    # t reads the one after the last chunk that ends at or before t ("post":
    # the chunk's last token reads its own chunk's update, the others the
    # chunk-start memory) or, "pre", the chunk-start memory.  There is no
    # Omega window on this path (c = 1) and Newton-Schulz, if any, is on the
    # momentum.  With C = 1 it is the per-token rule with c = 1.
    chunkwise = getattr(cfg, "update", "per_token") == "chunkwise"
    if chunkwise and (c != 1 or surprise_ns):
        raise ValueError("the chunk-wise update has no Omega window (c = 1) and no Newton-Schulz on the surprise")
    k = np.asarray(k, np.float64)
    q = np.asarray(q, np.float64)
    v = np.asarray(v, np.float64)
    T = k.shape[0]
    theta = np.asarray(theta, np.float64)
    eta = np.asarray(eta, np.float64)
    alpha = np.asarray(alpha, np.float64)
    gamma = np.ones(T) if gamma is None else np.asarray(gamma, np.float64)

    n_prev = 0 if cache_k is None else int(np.asarray(cache_k).shape[0])
    if n_prev:
        K_all = np.concatenate([np.asarray(cache_k, np.float64), k])
        V_all = np.concatenate([np.asarray(cache_v, np.float64), v])
        G_all = np.concatenate([np.asarray(cache_g, np.float64), gamma])
    else:
        K_all, V_all, G_all = k, v, gamma
    # row j + n_prev of the *_all arrays is token j of this call
    X_all = features(K_all, cfg.p, P)
    R = features(q, cfg.p, P)

    W = [np.array(m, np.float64) for m in W0]
    S = [np.array(m, np.float64) for m in S0]
    y = np.zeros((T, v.shape[1]))
    for s in range(0, T, C):
        e = min(s + C, T)
        W_bar = [m.copy() for m in W]
        lo = max(s - c + 1, -n_prev)               # oldest token any window reaches
        rows = slice(lo + n_prev, e + n_prev)
        grads = token_gradients(W_bar, X_all[rows], V_all[rows], depth)
        weighted = [g * G_all[rows][:, None, None] for g in grads]
        if chunkwise:
            # c = 1: the window rows are exactly the chunk's tokens s .. e-1
            G = [(wg * theta[s:e, None, None]).sum(axis=0) for wg in weighted]
            eta_bar, alpha_bar = eta[s:e].mean(), alpha[s:e].mean()
            S = [eta_bar * Sm - Gm for Sm, Gm in zip(S, G)]
            U = [newton_schulz(Sm, cfg.ns_iters) for Sm in S] if cfg.ns_iters else S
            W = [(1.0 - alpha_bar) * Wm + Um for Wm, Um in zip(W_bar, U)]
            y[s:e] = memory_apply(W_bar, R[s:e], depth)
            if not pre:
                y[e - 1] = memory_apply(W, R[e - 1:e], depth)[0]
            continue
        for t in range(s, e):
            first = max(t - c + 1, lo) - lo
            last = t - lo + 1
            g_t = [wg[first:last].sum(axis=0) for wg in weighted]
            if surprise_ns:
                # Newton-Schulz on the windowed surprise, eta and theta outside
                S = [eta[t] * Sm - theta[t] * newton_schulz(gm, cfg.ns_iters) for Sm, gm in zip(S, g_t)]
                U = S
            else:
                S = [eta[t] * Sm - theta[t] * gm for Sm, gm in zip(S, g_t)]
                U = [newton_schulz(Sm, cfg.ns_iters) for Sm in S] if cfg.ns_iters else S
            if pre:   # read-out with the memory before token t's update
                y[t] = memory_apply(W, R[t:t + 1], depth)[0]
            W = [(1.0 - alpha[t]) * Wm + Um for Wm, Um in zip(W, U)]
            if not pre:
                y[t] = memory_apply(W, R[t:t + 1], depth)[0]
    keep = min(c - 1, n_prev + T)
    cache = (K_all[len(K_all) - keep:], V_all[len(V_all) - keep:], G_all[len(G_all) - keep:])
    return y, W, S, cache


def _decode(a, dtype):
    if a is None:
        return None
    if dtype == "bf16" or np.asarray(a).dtype == np.uint16:
        return bf16_from_bits(a).astype(np.float64)
    return np.asarray(a, np.float64)


def unit_inputs(w, inp, u):
    """Decode the inputs of flattened unit u (= b*H + h) to fp64."""
    U = w.B * w.H

    def pick(a):
        if a is None:
            return None
        return np.asarray(a).reshape((U,) + np.asarray(a).shape[2:])[u]

    d = dict(
        k=_decode(pick(inp["k"]), w.qkv_dtype),
        q=_decode(pick(inp["q"]), w.qkv_dtype),
        v=_decode(pick(inp["v"]), w.qkv_dtype),
        theta=pick(inp["theta"]).astype(np.float64),
        eta=pick(inp["eta"]).astype(np.float64),
        alpha=pick(inp["alpha"]).astype(np.float64),
        gamma=None if inp["gamma"] is None else pick(inp["gamma"]).astype(np.float64),
        W0=[pick(m).astype(np.float64) for m in inp["W0"]],
        S0=[pick(m).astype(np.float64) for m in inp["S0"]],
        P=None if inp["P"] is None else _decode(inp["P"], "bf16"),
    )
    return d


def forward(w, inp, units=None, T=None):
    """Oracle over a list of units (default: all), optionally on the first T
    tokens only.  Returns dict(y [n, T, d_v], W [list of n x rows x cols],
    S [...], cache (k, v, gamma) lists)."""
    U = w.B * w.H
    units = range(U) if units is None else list(units)
    ys, Ws, Ss, caches = [], [], [], []
    for u in units:
        d = unit_inputs(w, inp, u)
        if T is not None:
            for key in ("k", "q", "v", "theta", "eta", "alpha", "gamma"):
                if d[key] is not None:
                    d[key] = d[key][:T]
        y, W, S, cache = forward_unit(w, d["k"], d["q"], d["v"], d["theta"], d["eta"],
                                      d["alpha"], d["gamma"], d["W0"], d["S0"], d["P"])
        ys.append(y)
        Ws.append(W)
        Ss.append(S)
        caches.append(cache)
    nm = len(Ws[0])
    return dict(
        y=np.stack(ys),
        W=[np.stack([W[m] for W in Ws]) for m in range(nm)],
        S=[np.stack([S[m] for S in Ss]) for m in range(nm)],
        cache=caches,
    )
