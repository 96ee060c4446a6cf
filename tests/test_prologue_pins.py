"""Pins of the fp64 oracle of the stage in front of the memory (projection,
short causal convolution, q/k normalisation, gate heads) against facts that
do not come from the oracle itself."""
import dataclasses
import os

import numpy as np
import pytest

from oracle.prologue import prologue_row
from tests import bruteforce as bf


@dataclasses.dataclass
class PCfg:
    H: int = 2
    d_k: int = 3
    d_v: int = 4
    conv: int = 4
    with_gamma: bool = True
    theta_max: float = 0.1


def _case(rng, cfg, T, D=5, cache=False):
    G = 4 if cfg.with_gamma else 3
    Nc = cfg.H * (2 * cfg.d_k + cfg.d_v)
    return dict(
        x=rng.standard_normal((T, D)),
        W_in=rng.standard_normal((D, Nc + G * cfg.H)) / np.sqrt(D),
        conv_w=rng.standard_normal((Nc, cfg.conv)) / 2.0,
        gate_b=rng.standard_normal((G, cfg.H)),
        cache=rng.standard_normal((cfg.conv - 1, Nc)) if cache else None,
    )


def _run(cfg, c):
    return prologue_row(cfg, c["x"], c["W_in"], c["conv_w"], c["gate_b"], c["cache"])


@pytest.mark.parametrize("with_gamma,cache,K", [(True, False, 4), (False, True, 4), (True, True, 2), (False, False, 1)])
def test_matches_scalar_loops(with_gamma, cache, K):
    cfg = PCfg(with_gamma=with_gamma, conv=K)
    rng = np.random.default_rng(10 + K + 2 * with_gamma + cache)
    c = _case(rng, cfg, T=7, cache=cache)
    o = _run(cfg, c)
    b = bf.prologue(cfg.H, cfg.d_k, cfg.d_v, K, with_gamma, cfg.theta_max, c["x"].tolist(), c["W_in"].tolist(),
                    c["conv_w"].tolist(), c["gate_b"].tolist(), None if c["cache"] is None else c["cache"].tolist())
    for key in ("q", "k", "v", "theta", "eta", "alpha", "gamma", "cache"):
        if o[key] is None:
            assert b[key] is None
            continue
        np.testing.assert_allclose(o[key], np.array(b[key]).reshape(o[key].shape), rtol=1e-12, atol=1e-13)


def test_convolution_is_numpy_convolve_per_channel():
    """v is the convolved projection without normalisation: per channel it is
    numpy's full convolution of the channel with the reversed taps, cut to T."""
    cfg = PCfg(with_gamma=False)
    rng = np.random.default_rng(21)
    c = _case(rng, cfg, T=9)
    o = _run(cfg, c)
    u = c["x"] @ c["W_in"]
    base = 2 * cfg.H * cfg.d_k
    for h in range(cfg.H):
        for i in range(cfg.d_v):
            ch = base + h * cfg.d_v + i
            ref = np.convolve(u[:, ch], c["conv_w"][ch][::-1])[:9]
            np.testing.assert_allclose(o["v"][h, :, i], ref, rtol=1e-12, atol=1e-13)


def test_identity_taps_give_normalised_projections():
    """With the taps e_{K-1} the convolution is the identity: q and k are the
    unit-normalised head slices of x W_in, v the raw slice."""
    cfg = PCfg()
    rng = np.random.default_rng(22)
    c = _case(rng, cfg, T=6)
    c["conv_w"] = np.zeros_like(c["conv_w"])
    c["conv_w"][:, -1] = 1.0
    o = _run(cfg, c)
    u = c["x"] @ c["W_in"]
    for h in range(cfg.H):
        qh = u[:, h * cfg.d_k:(h + 1) * cfg.d_k]
        np.testing.assert_allclose(o["q"][h], qh / np.linalg.norm(qh, axis=1, keepdims=True), rtol=1e-12)
        vh = u[:, 2 * cfg.H * cfg.d_k + h * cfg.d_v:2 * cfg.H * cfg.d_k + (h + 1) * cfg.d_v]
        np.testing.assert_allclose(o["v"][h], vh, rtol=1e-12)


def test_unit_norms_and_zero_input():
    """q and k have unit norm; with x = 0 they are exactly zero (no division
    by zero) and every gate is its sigmoid of the bias."""
    cfg = PCfg()
    rng = np.random.default_rng(23)
    c = _case(rng, cfg, T=5)
    o = _run(cfg, c)
    np.testing.assert_allclose(np.linalg.norm(o["q"], axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(np.linalg.norm(o["k"], axis=-1), 1.0, rtol=1e-13)
    c["x"] = np.zeros_like(c["x"])
    o = _run(cfg, c)
    assert not np.any(o["q"]) and not np.any(o["k"]) and not np.any(o["v"])
    sig = 1.0 / (1.0 + np.exp(-c["gate_b"]))
    np.testing.assert_allclose(o["theta"], np.repeat(0.1 * sig[0][:, None], 5, axis=1), rtol=1e-14)
    np.testing.assert_allclose(o["alpha"], np.repeat(sig[2][:, None], 5, axis=1), rtol=1e-14)


def test_causal_reach_of_one_token():
    """Changing x_j changes q, k, v exactly at tokens j .. j+K-1 and the
    gates only at token j."""
    cfg = PCfg()
    rng = np.random.default_rng(24)
    c = _case(rng, cfg, T=12)
    a = _run(cfg, c)
    j = 4
    c["x"][j] += rng.standard_normal(c["x"].shape[1])
    b = _run(cfg, c)
    for key in ("q", "k", "v"):
        moved = np.abs(a[key] - b[key]).max(axis=(0, 2)) > 1e-12
        assert moved.tolist() == [j <= t < j + cfg.conv for t in range(12)], key
    for key in ("theta", "eta", "alpha", "gamma"):
        moved = np.abs(a[key] - b[key]).max(axis=0) > 1e-15
        assert moved.tolist() == [t == j for t in range(12)], key


@pytest.mark.parametrize("T1", [2, 5])
def test_split_with_carried_cache(T1):
    """Two calls with the carried convolution cache equal one call, also when
    the first call is shorter than the cache."""
    cfg = PCfg()
    rng = np.random.default_rng(25 + T1)
    c = _case(rng, cfg, T=10, cache=True)
    whole = _run(cfg, c)
    first = dict(c, x=c["x"][:T1])
    o1 = _run(cfg, first)
    o2 = _run(cfg, dict(c, x=c["x"][T1:], cache=o1["cache"]))
    for key in ("q", "k", "v", "theta", "eta", "alpha", "gamma"):
        np.testing.assert_allclose(np.concatenate([o1[key], o2[key]], axis=1), whole[key], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(o2["cache"], whole["cache"], rtol=1e-14)


def test_hand_worked_golden():
    """A 1-wide model worked by hand (tests/golden/prologue_scalar.txt):
    column order, tap orientation, normalisation, gate biases, theta_max and
    the outgoing cache."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "prologue_scalar.txt")
    taps, outs = [], {}
    for ln in open(path):
        if ln.startswith("#") or not ln.strip():
            continue
        head, vals = ln.split(":")
        nums = [float(t) for t in vals.split()]
        if head == "win":
            W_in = np.array([nums])
        elif head.startswith("tap"):
            taps.append(nums)
        elif head == "bias":
            gate_b = np.array(nums)[:, None]
        elif head == "x":
            x = np.array(nums)[:, None]
        else:
            outs[head.split()[1]] = np.array(nums)
    cfg = PCfg(H=1, d_k=2, d_v=1, conv=2, with_gamma=False)
    o = prologue_row(cfg, x, W_in, np.array(taps), gate_b)
    np.testing.assert_allclose(o["q"].ravel(), outs["q"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(o["k"].ravel(), outs["k"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(o["v"].ravel(), outs["v"], rtol=0, atol=1e-15)
    for g in ("theta", "eta", "alpha"):
        np.testing.assert_allclose(o[g].ravel(), outs[g], rtol=1e-15, atol=0)
    assert o["gamma"] is None
    np.testing.assert_allclose(o["cache"].ravel(), outs["cache"], rtol=0, atol=0)
