"""A second, deliberately different CPU reference used only to pin the oracle.

It shares nothing with ``oracle/``:

* monomials come from ``itertools.combinations_with_replacement`` with a
  1/m! coefficient computed from the multiset's size;
* per-token gradients come from torch autograd on the scalar loss
  ||M_W(x_i) - v_i||^2 (no hand-written chain rule);
* Newton-Schulz is evaluated through its closed form: for X/(||X||_F + eps) =
  U diag(s) V^T, k quintic steps give U diag(f^k(s)) V^T with
  f(s) = a s + b s^3 + c s^5 (every step maps singular values through f and
  keeps the singular vectors);
* everything is a plain per-token loop over python lists.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch

QUINTIC = (3.4445, -4.7750, 2.0315)
EPS = 1e-7


def monomials(x, p):
    x = [float(t) for t in x]
    if p == 1:
        return np.array(x)
    out = []
    for m in range(p + 1):
        for combo in itertools.combinations_with_replacement(range(len(x)), m):
            val = 1.0 / math.factorial(m)
            for i in combo:
                val *= x[i]
            out.append(val)
    return np.array(out)


def ns_closed_form(G, k):
    G = np.asarray(G, np.float64)
    X = G / (np.linalg.norm(G) + EPS)
    U, s, Vt = np.linalg.svd(X, full_matrices=False)
    a, b, c = QUINTIC
    for _ in range(k):
        s = a * s + b * s ** 3 + c * s ** 5
    return (U * s) @ Vt


def _mem(Wt, x, depth):
    if depth == 1:
        return x @ Wt[0]
    z = x @ Wt[0]
    return x + torch.nn.functional.silu(z) @ Wt[1]


def autograd_grad(W, x, v, depth):
    Wt = [torch.tensor(m, dtype=torch.float64, requires_grad=True) for m in W]
    xt = torch.tensor(x, dtype=torch.float64)
    vt = torch.tensor(v, dtype=torch.float64)
    loss = ((_mem(Wt, xt, depth) - vt) ** 2).sum()
    gs = torch.autograd.grad(loss, Wt)
    return [g.numpy() for g in gs]


def apply_mem(W, x, depth):
    with torch.no_grad():
        Wt = [torch.tensor(m, dtype=torch.float64) for m in W]
        return _mem(Wt, torch.tensor(x, dtype=torch.float64), depth).numpy()


def forward(depth, C, c, p, ns_iters, k, q, v, theta, eta, alpha, gamma, W0, S0,
            P=None, prev=None, pre=False, surprise_ns=False, chunkwise=False):
    """prev = (keys, values, gammas) of tokens preceding the call, oldest first.
    pre = True reads token t out of the memory before its update (the paper's
    MAC retrieval, h_t = M*_{t-1}(q_t)); else after it.  surprise_ns = True
    orthogonalises each token's windowed gradient instead of the momentum.
    chunkwise = True runs the chunk-wise store path instead (no window)."""
    T = len(k)
    gamma = np.ones(T) if gamma is None else gamma
    pk, pv, pg = ([], [], []) if prev is None else prev
    keys = list(pk) + list(k)
    vals = list(pv) + list(v)
    gams = list(pg) + list(gamma)
    n_prev = len(pk)

    def feat(vec):
        f = monomials(vec, p)
        return f if P is None else f @ np.asarray(P, np.float64)

    W = [np.array(m, np.float64) for m in W0]
    S = [np.array(m, np.float64) for m in S0]
    if chunkwise:
        return _chunkwise(depth, C, ns_iters, feat, keys, vals, gams, n_prev, q, theta, eta, alpha, W, S, pre)
    W_bar = None
    y = []
    for t in range(T):
        if t % C == 0:
            W_bar = [m.copy() for m in W]
        g = [np.zeros_like(m) for m in W]
        for i in range(t - c + 1, t + 1):
            if i < -n_prev:
                continue
            gi = autograd_grad(W_bar, feat(keys[i + n_prev]), np.asarray(vals[i + n_prev]), depth)
            g = [a + gams[i + n_prev] * b for a, b in zip(g, gi)]
        if surprise_ns and ns_iters:
            S = [eta[t] * Sm - theta[t] * ns_closed_form(gm, ns_iters) for Sm, gm in zip(S, g)]
            U = S
        else:
            S = [eta[t] * Sm - theta[t] * gm for Sm, gm in zip(S, g)]
            U = [ns_closed_form(Sm, ns_iters) for Sm in S] if ns_iters else S
        W_before = W
        W = [(1.0 - alpha[t]) * Wm + Um for Wm, Um in zip(W, U)]
        y.append(apply_mem(W_before if pre else W, feat(q[t]), depth))
    return np.array(y), W, S


def _chunkwise(depth, C, ns_iters, feat, keys, vals, gams, n_prev, q, theta, eta, alpha, W, S, pre):
    """Chunk-wise store path, written as loops: per chunk one gradient summed
    over its tokens at the chunk-start memory (each token's weighted by its
    theta and gamma), one momentum step with the chunk's average eta, one
    decay step with its average alpha; a token reads the memory after the
    last chunk that has ended by it (or, pre, its chunk's start memory)."""
    T = len(q)
    y = []
    for s in range(0, T, C):
        e = min(s + C, T)
        W_bar = W
        G = [np.zeros_like(m) for m in W]
        eta_sum = alpha_sum = 0.0
        for i in range(s, e):
            gi = autograd_grad(W_bar, feat(keys[i + n_prev]), np.asarray(vals[i + n_prev]), depth)
            G = [a + theta[i] * gams[i + n_prev] * b for a, b in zip(G, gi)]
            eta_sum += eta[i]
            alpha_sum += alpha[i]
        n = e - s
        S = [(eta_sum / n) * Sm - Gm for Sm, Gm in zip(S, G)]
        U = [ns_closed_form(Sm, ns_iters) for Sm in S] if ns_iters else S
        W = [(1.0 - alpha_sum / n) * Wm + Um for Wm, Um in zip(W_bar, U)]
        for t in range(s, e):
            reads = W if (t == e - 1 and not pre) else W_bar
            y.append(apply_mem(reads, feat(q[t]), depth))
    return np.array(y), W, S


def prologue(H, d_k, d_v, K, with_gamma, theta_max, x, W_in, conv_w, gate_b, cache=None):
    """The stage in front of the memory as scalar loops: every projected
    channel is a dot product over the model width, the convolution walks its
    taps backwards in time, norms are square roots of explicit sums, and the
    sigmoid is math.exp.  Returns per head lists of q, k, v rows and gate
    values, and the outgoing cache rows."""
    T, D = len(x), len(x[0])
    N = len(W_in[0])
    Nc = H * (2 * d_k + d_v)
    G = 4 if with_gamma else 3
    u = [[sum(float(x[t][i]) * float(W_in[i][n]) for i in range(D)) for n in range(N)] for t in range(T)]
    past = [[0.0] * Nc for _ in range(K - 1)] if cache is None else [[float(a) for a in row] for row in cache]
    rows = past + [r[:Nc] for r in u]

    def conv(t, c):
        return sum(float(conv_w[c][K - 1 - j]) * rows[K - 1 + t - j][c] for j in range(K))

    out = {"q": [], "k": [], "v": []}
    for h in range(H):
        for name, base, d, norm in (("q", h * d_k, d_k, True), ("k", H * d_k + h * d_k, d_k, True),
                                    ("v", 2 * H * d_k + h * d_v, d_v, False)):
            seq = []
            for t in range(T):
                vec = [conv(t, base + i) for i in range(d)]
                if norm:
                    n2 = math.sqrt(sum(a * a for a in vec))
                    vec = [a / max(n2, 1e-12) for a in vec]
                seq.append(vec)
            out[name].append(seq)
    for g, name in enumerate(("theta", "eta", "alpha", "gamma")):
        if g >= G:
            out[name] = None
            continue
        out[name] = [[(theta_max if name == "theta" else 1.0)
                      / (1.0 + math.exp(-(u[t][Nc + g * H + h] + float(gate_b[g][h])))) for t in range(T)]
                     for h in range(H)]
    out["cache"] = rows[len(rows) - (K - 1):]
    return out
