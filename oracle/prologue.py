"""Plain fp64 oracle of the stage in front of the memory: projections, short
causal convolution, q/k normalisation and the gate heads.

TEST INFRASTRUCTURE ONLY: used by ``tests/`` and ``bench.py``'s CPU legs;
never by the library.  It shares no code with the CUDA path.

For one batch row, token by token:

* projection  u_t = x_t W_in, one matrix whose columns are the query heads,
              the key heads, the value heads, then one logit column per head
              for each gate (theta, eta, alpha, and gamma where the Omega
              weights are produced).  The titans-torch 0.1.2 project page
              (API Reference, TitansMAC forward flow: q = W_Q S) and the
              NeuralMemory usage of the atlas-torch README ("Configuration":
              the memory takes the model-width sequence) put the
              projections here.
* short conv  the q, k and v channels go through a causal depthwise
              convolution of K taps (the atlas-torch README, "Atlas
              Extensions": CausalDepthwiseConv1d with kernel 4 on keys,
              values and queries): conv_t[c] = sum_{j<K} w[c][K-1-j] u_{t-j}[c],
              rows before the call from the carried cache (zeros at the start
              of the sequence); no bias.
* normalise   each head's query and key are divided by their L2 norm
              (x / max(|x|, 1e-12), so a zero vector stays zero).
* gates       theta = theta_max sigmoid(l + b), eta, alpha, gamma =
              sigmoid(l + b), with l the head's logit column and b its bias
              (titans-torch 0.1.2 project page, API Reference, the
              inner-loop update rule: alpha, theta, eta come from the data
              through small networks; a linear head is the smallest).
"""
from __future__ import annotations

import numpy as np

GATES = ("theta", "eta", "alpha", "gamma")
NORM_EPS = 1e-12


def prologue_row(cfg, x, W_in, conv_w, gate_b, cache=None):
    """One batch row.

    cfg: H, d_k, d_v, conv (K), with_gamma, theta_max.
    x [T, D]; W_in [D, N]; conv_w [Nc, K]; gate_b [G, H]; cache [K-1, Nc] or
    None (the projected q/k/v rows before this call, oldest first).
    Returns dict(q [H, T, d_k], k, v [H, T, d_v], theta [H, T], eta, alpha,
    gamma (or None), cache [K-1, Nc])."""
    H, dk, dv, K = cfg.H, cfg.d_k, cfg.d_v, cfg.conv
    G = 4 if cfg.with_gamma else 3
    Nc = H * (2 * dk + dv)
    x = np.asarray(x, np.float64)
    W_in = np.asarray(W_in, np.float64)
    conv_w = np.asarray(conv_w, np.float64)
    gate_b = np.asarray(gate_b, np.float64)
    T = x.shape[0]
    assert W_in.shape[1] == Nc + G * H
    u = x @ W_in
    prev = np.zeros((K - 1, Nc)) if cache is None else np.asarray(cache, np.float64)
    uc = np.concatenate([prev, u[:, :Nc]])          # row K-1+t is token t
    conv = np.zeros((T, Nc))
    for t in range(T):
        for j in range(K):
            conv[t] += conv_w[:, K - 1 - j] * uc[K - 1 + t - j]
    out = {}
    for name, off, d, norm in (("q", 0, dk, True), ("k", H * dk, dk, True), ("v", 2 * H * dk, dv, False)):
        a = conv[:, off:off + H * d].reshape(T, H, d).transpose(1, 0, 2)
        if norm:
            a = a / np.maximum(np.linalg.norm(a, axis=-1, keepdims=True), NORM_EPS)
        out[name] = a
    for gi, name in enumerate(GATES):
        if gi >= G:
            out[name] = None
            continue
        logit = u[:, Nc + gi * H:Nc + (gi + 1) * H] + gate_b[gi]
        s = 1.0 / (1.0 + np.exp(-logit))
        out[name] = (cfg.theta_max * s if name == "theta" else s).T
    out["cache"] = uc[len(uc) - (K - 1):] if K > 1 else np.zeros((0, Nc))
    return out
