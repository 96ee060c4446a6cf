"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

Each test names the passage it follows.  None of them re-types the oracle's
own formulas: they use hand-worked values, finite differences, autograd,
closed forms, invariants, or the independent per-token reference in
``tests/bruteforce.py``.
"""
import dataclasses
import itertools
import math
import os

import numpy as np
import pytest

import oracle
from tests import bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@dataclasses.dataclass
class Cfg:
    depth: int = 1
    C: int = 4
    c: int = 1
    p: int = 1
    ns_iters: int = 0
    readout: str = "post"
    ns_target: str = "momentum"
    update: str = "per_token"


def _rand_case(rng, depth, d_k, d_v, hidden, T, p=1, proj=0, gamma=True, scale_w=0.3):
    k = rng.standard_normal((T, d_k))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((T, d_k))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    v = rng.standard_normal((T, d_v))
    theta = 0.1 / (1 + np.exp(-rng.standard_normal(T)))
    eta = 1 / (1 + np.exp(-rng.normal(1, 1, T)))
    alpha = 1 / (1 + np.exp(-rng.normal(-3, 1, T)))
    g = 1 / (1 + np.exp(-rng.standard_normal(T))) if gamma else None
    F = d_k if p == 1 else math.comb(d_k + 2, 2)
    P = rng.standard_normal((F, proj)) / np.sqrt(F) if proj else None
    Fm = proj if proj else F
    if depth == 1:
        shapes = [(Fm, d_v)]
    else:
        shapes = [(Fm, hidden), (hidden, d_v)]
    W0 = [scale_w * rng.standard_normal(s) for s in shapes]
    S0 = [0.1 * rng.standard_normal(s) for s in shapes]
    return dict(k=k, q=q, v=v, theta=theta, eta=eta, alpha=alpha, gamma=g, W0=W0, S0=S0, P=P)


def _run_oracle(cfg, case, cache=None):
    kw = {}
    if cache is not None:
        kw = dict(cache_k=cache[0], cache_v=cache[1], cache_g=cache[2])
    return oracle.forward_unit(cfg, case["k"], case["q"], case["v"], case["theta"], case["eta"],
                               case["alpha"], case["gamma"], case["W0"], case["S0"], case["P"], **kw)


# ------------------------------------------------------------ feature map
def test_poly_golden_worked_example():
    """atlas-torch README, "Atlas Extensions": Polynomial Features."""
    lines = [ln for ln in open(os.path.join(GOLDEN, "poly_features_d3.txt")) if not ln.startswith("#")]
    x = np.array([float(t) for t in lines[0].split(":")[1].split()])
    want = np.array([float(t) for t in lines[1].split(":")[1].split()])
    got = oracle.poly_features(x[None], 2)[0]
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("d", [1, 3, 7])
def test_poly_matches_itertools_enumeration(d):
    """Exact monomial expansion with 1/m! (atlas-torch README, Polynomial Features)."""
    x = np.random.default_rng(d).standard_normal(d)
    np.testing.assert_allclose(oracle.poly_features(x[None], 2)[0], bf.monomials(x, 2), rtol=0, atol=1e-15)


@pytest.mark.parametrize("d,width", [(32, 561), (64, 2145), (5, 21)])
def test_poly_width(d, width):
    """1 + d + d(d+1)/2 monomials; 561 for 32-dim keys (ATLAS summary, Section 3.1)."""
    assert oracle.poly_features(np.zeros((1, d)), 2).shape[1] == width == math.comb(d + 2, 2)


def test_poly_kernel_identity():
    """phi(x).phi(y) = 1 + x.y + ((x.y)^2 + sum x_i^2 y_i^2)/8 for the 1/m! map."""
    rng = np.random.default_rng(7)
    for d in (4, 32):
        x, y = rng.standard_normal((2, d))
        lhs = oracle.poly_features(x[None], 2)[0] @ oracle.poly_features(y[None], 2)[0]
        xy = x @ y
        rhs = 1 + xy + (xy ** 2 + np.sum(x ** 2 * y ** 2)) / 8
        assert abs(lhs - rhs) < 1e-12 * max(1, abs(rhs))


def test_projection_is_applied_after_expansion():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 4))
    P = rng.standard_normal((15, 3))
    want = np.stack([bf.monomials(r, 2) @ P for r in x])
    np.testing.assert_allclose(oracle.features(x, 2, P), want, rtol=1e-13, atol=1e-13)


# -------------------------------------------------------------- gradients
def _fd_grad(W, x, v, depth, h=1e-6):
    out = []
    for m in range(len(W)):
        g = np.zeros_like(W[m])
        for idx in itertools.product(*[range(s) for s in W[m].shape]):
            Wp = [w.copy() for w in W]
            Wm = [w.copy() for w in W]
            Wp[m][idx] += h
            Wm[m][idx] -= h
            lp = np.sum((oracle.memory_apply(Wp, x[None], depth)[0] - v) ** 2)
            lm = np.sum((oracle.memory_apply(Wm, x[None], depth)[0] - v) ** 2)
            g[idx] = (lp - lm) / (2 * h)
        out.append(g)
    return out


@pytest.mark.parametrize("depth", [1, 2])
def test_gradient_matches_finite_differences(depth):
    """Gradient of Eq. 12 (titans-pytorch-mlx README) by central differences."""
    rng = np.random.default_rng(depth)
    d, h = 3, 4
    x, v = rng.standard_normal(d), rng.standard_normal(d)
    W = [rng.standard_normal((d, d))] if depth == 1 else [rng.standard_normal((d, h)), rng.standard_normal((h, d))]
    got = oracle.token_gradients(W, x[None], v[None], depth)
    want = _fd_grad(W, x, v, depth)
    for g, w in zip(got, want):
        np.testing.assert_allclose(g[0], w, rtol=1e-7, atol=1e-8)


@pytest.mark.parametrize("depth", [1, 2])
def test_gradient_matches_autograd(depth):
    rng = np.random.default_rng(10 + depth)
    d, h, n = 5, 7, 6
    X, V = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    W = [rng.standard_normal((d, d))] if depth == 1 else [rng.standard_normal((d, h)), rng.standard_normal((h, d))]
    got = oracle.token_gradients(W, X, V, depth)
    for i in range(n):
        want = bf.autograd_grad(W, X[i], V[i], depth)
        for g, w in zip(got, want):
            np.testing.assert_allclose(g[i], w, rtol=1e-12, atol=1e-12)


def test_linear_gradient_is_delta_rule_outer_product():
    """Linear memory: the gradient is (prediction error) x (key), scaled by 2
    (atlas-torch README, "How the memory works"), checked by differences of
    the loss along rank-1 probes."""
    rng = np.random.default_rng(5)
    d_k, d_v = 4, 3
    x, v, W = rng.standard_normal(d_k), rng.standard_normal(d_v), rng.standard_normal((d_k, d_v))
    g = oracle.token_gradients([W], x[None], v[None], 1)[0][0]
    assert np.linalg.matrix_rank(g, tol=1e-10) == 1
    # the column space is the key, the row space the prediction error
    err = x @ W - v
    np.testing.assert_allclose(np.abs(g @ err) / np.linalg.norm(g @ err), np.abs(x) / np.linalg.norm(x), atol=1e-12)


# -------------------------------------------------------- whole recurrence
def _golden_scalar():
    rows, cases = [], {}
    for ln in open(os.path.join(GOLDEN, "titans_scalar_1d.txt")):
        if ln.startswith("#") or not ln.strip():
            continue
        if ln.startswith("tok"):
            rows.append([float(t) for t in ln.split(":")[1].split()])
        elif ln.startswith("case"):
            head, vals = ln.split(":")
            _, name, what = head.split()
            cases.setdefault(name, {})[what] = np.array([float(t) for t in vals.split()])
    return np.array(rows), cases


@pytest.mark.parametrize("name,C,c,use_gamma", [("C1c1", 1, 1, False), ("C2c1", 2, 1, False), ("C2c2", 2, 2, True)])
def test_hand_worked_scalar_memory(name, C, c, use_gamma):
    """Values worked by hand from Eq. 12-14 (titans-pytorch-mlx README)."""
    rows, cases = _golden_scalar()
    k, v, q, theta, eta, alpha, gamma = rows.T
    y, W, S, _ = oracle.forward_unit(Cfg(depth=1, C=C, c=c), k[:, None], q[:, None], v[:, None], theta, eta,
                                     alpha, gamma if use_gamma else None, [np.array([[0.5]])], [np.zeros((1, 1))])
    np.testing.assert_allclose(y[:, 0], cases[name]["y"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(W[0].ravel(), cases[name]["W"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(S[0].ravel(), cases[name]["S"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("name,readout,use_gamma", [("CW2", "post", False), ("CW2pre", "pre", False),
                                                    ("CW2g", "post", True)])
def test_hand_worked_scalar_memory_chunkwise(name, readout, use_gamma):
    """The chunk-wise rule on the same three tokens, worked by hand (C = 2,
    so the last token is a partial chunk of its own)."""
    rows, cases = _golden_scalar()
    k, v, q, theta, eta, alpha, gamma = rows.T
    y, W, S, _ = oracle.forward_unit(Cfg(depth=1, C=2, c=1, readout=readout, update="chunkwise"), k[:, None],
                                     q[:, None], v[:, None], theta, eta, alpha, gamma if use_gamma else None,
                                     [np.array([[0.5]])], [np.zeros((1, 1))])
    np.testing.assert_allclose(y[:, 0], cases[name]["y"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(W[0].ravel(), cases[name]["W"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(S[0].ravel(), cases[name]["S"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("depth", [1, 2])
def test_C1_is_the_sequential_titans_rule(depth):
    """C = 1: every token sees the weights left by the token before, i.e. the
    sequential update of Eq. 13-14 (titans-pytorch-mlx README)."""
    rng = np.random.default_rng(20 + depth)
    case = _rand_case(rng, depth, 4, 4, 6, T=9)
    y, W, S, _ = _run_oracle(Cfg(depth=depth, C=1, c=1), case)
    yb, Wb, Sb = bf.forward(depth, 1, 1, 1, 0, case["k"], case["q"], case["v"], case["theta"], case["eta"],
                            case["alpha"], case["gamma"], case["W0"], case["S0"])
    np.testing.assert_allclose(y, yb, rtol=1e-11, atol=1e-12)
    for a, b in zip(W + S, Wb + Sb):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_window_of_one_is_the_single_token_update():
    """c = 1 recovers the single-association update (ATLAS summary, Section 3.2):
    with a window of one, token t's surprise is gamma_t times its own gradient
    only, which we check against the per-token reference at C = 4."""
    rng = np.random.default_rng(31)
    case = _rand_case(rng, 2, 3, 3, 5, T=10)
    y, W, S, _ = _run_oracle(Cfg(depth=2, C=4, c=1), case)
    yb, Wb, Sb = bf.forward(2, 4, 1, 1, 0, case["k"], case["q"], case["v"], case["theta"], case["eta"],
                            case["alpha"], case["gamma"], case["W0"], case["S0"])
    np.testing.assert_allclose(y, yb, rtol=1e-11, atol=1e-12)
    for a, b in zip(W + S, Wb + Sb):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("ns", [0, 5])
def test_alpha_one_wipes_the_state(ns):
    """alpha_t = 1 forgets everything: W_t = U_t (Eq. 13)."""
    rng = np.random.default_rng(40 + ns)
    case = _rand_case(rng, 2, 4, 4, 6, T=5)
    case["alpha"] = np.ones(5)
    y, W, S, _ = _run_oracle(Cfg(depth=2, C=2, c=2, ns_iters=ns), case)
    for Wm, Sm in zip(W, S):
        want = bf.ns_closed_form(Sm, ns) if ns else Sm
        np.testing.assert_allclose(Wm, want, rtol=1e-11, atol=1e-12)


def test_closed_form_without_momentum_or_decay():
    """eta = alpha = 0, one chunk, no Newton-Schulz, linear memory:
    W_T = W0 - sum_t theta_t 2 x_t^T (x_t W0 - v_t)."""
    rng = np.random.default_rng(50)
    T = 12
    case = _rand_case(rng, 1, 5, 3, 0, T=T, gamma=False)
    case["eta"], case["alpha"] = np.zeros(T), np.zeros(T)
    y, W, S, _ = _run_oracle(Cfg(depth=1, C=T, c=1), case)
    X, V, W0 = case["k"], case["v"], case["W0"][0]
    closed = W0 - np.einsum("t,ti,tj->ij", 2 * case["theta"], X, X @ W0 - V)
    np.testing.assert_allclose(W[0], closed, rtol=1e-12, atol=1e-13)
    # and the read-out uses the post-update weights of each token
    partial = W0 - np.cumsum(np.einsum("t,ti,tj->tij", 2 * case["theta"], X, X @ W0 - V), axis=0)
    np.testing.assert_allclose(y, np.einsum("ti,tij->tj", case["q"], partial), rtol=1e-12, atol=1e-13)


def test_window_perturbation_reaches_exactly_the_next_c_tokens():
    """The Omega window of token t covers tokens t-c+1..t (atlas-torch README,
    "Bug Fixes": Omega window slide).  With eta = 0 and alpha = 1 the read-out
    of token t depends on the surprise g_t alone, so perturbing v_j must move
    y_t for t in [j, j+c-1] and nowhere else (one chunk, weights frozen)."""
    rng = np.random.default_rng(60)
    T, c = 16, 4
    case = _rand_case(rng, 1, 4, 3, 0, T=T)
    case["eta"], case["alpha"] = np.zeros(T), np.ones(T)
    cfg = Cfg(depth=1, C=T, c=c)
    y0 = _run_oracle(cfg, case)[0]
    for j in (0, 5, 13):
        pert = dict(case, v=case["v"].copy())
        pert["v"][j] += 1.0
        moved = np.abs(_run_oracle(cfg, pert)[0] - y0).max(axis=1) > 1e-12
        assert list(np.nonzero(moved)[0]) == list(range(j, min(T, j + c)))


# ------------------------------------------------------------ Newton-Schulz
def test_ns_matches_svd_closed_form():
    """Each quintic step maps singular values through f and keeps the singular
    vectors; compare with the SVD form for wide, tall and square inputs."""
    rng = np.random.default_rng(70)
    for shape in [(6, 11), (11, 6), (7, 7)]:
        G = rng.standard_normal(shape) * 3.0
        for k in (1, 3, 5):
            np.testing.assert_allclose(oracle.newton_schulz(G, k), bf.ns_closed_form(G, k), rtol=1e-10, atol=1e-12)


def test_ns_invariances_and_rank_one():
    rng = np.random.default_rng(71)
    G = rng.standard_normal((8, 20))
    # positive scale invariance (up to eps) and odd symmetry
    np.testing.assert_allclose(oracle.newton_schulz(7.0 * G, 5), oracle.newton_schulz(G, 5), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(oracle.newton_schulz(-G, 5), -oracle.newton_schulz(G, 5), rtol=0, atol=1e-14)
    assert np.all(oracle.newton_schulz(np.zeros((3, 5)), 5) == 0)
    # rank one: singular value s = |G|/(|G| + eps) goes through f five times
    u, v = rng.standard_normal(8), rng.standard_normal(20)
    R1 = np.outer(u, v)
    s = np.linalg.norm(R1) / (np.linalg.norm(R1) + 1e-7)
    for _ in range(5):
        s = 3.4445 * s - 4.7750 * s ** 3 + 2.0315 * s ** 5
    out = oracle.newton_schulz(R1, 5)
    assert abs(np.linalg.svd(out, compute_uv=False)[0] - s) < 1e-12
    assert abs(s - 0.69644) < 5e-5
    assert np.linalg.matrix_rank(out, tol=1e-9) == 1


def test_ns_output_is_near_orthogonal():
    """Momentum is made approximately semi-orthogonal (ATLAS summary, Section 5):
    normalised singular values >= 0.05 land in [0.68, 1.13] after 5 steps."""
    rng = np.random.default_rng(72)
    U, _ = np.linalg.qr(rng.standard_normal((16, 16)))
    V, _ = np.linalg.qr(rng.standard_normal((40, 16)))
    s = np.linspace(0.05, 0.4, 16)
    s = s / np.linalg.norm(s)        # Frobenius norm 1, smallest value > 0.05
    assert s.min() >= 0.05
    G = (U * s) @ V.T
    out_s = np.linalg.svd(oracle.newton_schulz(G, 5), compute_uv=False)
    assert out_s.min() > 0.68 - 1e-9 and out_s.max() < 1.13 + 1e-9


# ---------------------------------------------------- continuation, general
@pytest.mark.parametrize("depth,c,ns", [(1, 3, 0), (2, 4, 0), (2, 3, 3)])
def test_split_continuation(depth, c, ns):
    """Chunked inference with carried state equals the whole-sequence forward
    (atlas-torch README, "Status and scope", limitation 5)."""
    rng = np.random.default_rng(80 + depth + c)
    T, T1, C = 24, 8, 4
    case = _rand_case(rng, depth, 4, 4, 6, T=T)
    cfg = Cfg(depth=depth, C=C, c=c, ns_iters=ns)
    y, W, S, _ = _run_oracle(cfg, case)
    first = {k: (v[:T1] if isinstance(v, np.ndarray) and v.shape[:1] == (T,) else v) for k, v in case.items()}
    y1, W1, S1, cache = _run_oracle(cfg, first)
    second = {k: (v[T1:] if isinstance(v, np.ndarray) and v.shape[:1] == (T,) else v) for k, v in case.items()}
    second["W0"], second["S0"] = W1, S1
    y2, W2, S2, _ = _run_oracle(cfg, second, cache=cache)
    np.testing.assert_allclose(np.concatenate([y1, y2]), y, rtol=1e-12, atol=1e-12)
    for a, b in zip(W2 + S2, W + S):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


BRUTE_CASES = [
    # depth, C, c, p, proj, ns, d_k, d_v, hidden, T
    (1, 4, 1, 1, 0, 0, 4, 3, 0, 10),
    (2, 4, 1, 1, 0, 0, 4, 4, 6, 10),
    (1, 4, 3, 2, 0, 0, 3, 2, 0, 11),      # Omega + polynomial features
    (1, 3, 5, 2, 0, 0, 2, 2, 0, 9),       # window longer than a chunk
    (2, 4, 3, 1, 0, 5, 4, 4, 6, 10),      # Omega + Muon
    (2, 4, 3, 2, 4, 5, 3, 4, 5, 9),       # polynomial + projection + Muon
]


@pytest.mark.parametrize("case_def", BRUTE_CASES)
def test_oracle_matches_independent_bruteforce(case_def):
    depth, C, c, p, proj, ns, d_k, d_v, hidden, T = case_def
    rng = np.random.default_rng(hash(case_def) % 2 ** 32)
    case = _rand_case(rng, depth, d_k, d_v, hidden, T, p=p, proj=proj)
    cfg = Cfg(depth=depth, C=C, c=c, p=p, ns_iters=ns)
    y, W, S, _ = _run_oracle(cfg, case)
    yb, Wb, Sb = bf.forward(depth, C, c, p, ns, case["k"], case["q"], case["v"], case["theta"], case["eta"],
                            case["alpha"], case["gamma"], case["W0"], case["S0"], case["P"])
    np.testing.assert_allclose(y, yb, rtol=1e-10, atol=1e-11)
    for a, b in zip(W + S, Wb + Sb):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


def test_bruteforce_with_window_cache():
    """Windows reach back into tokens handed over from a previous call."""
    rng = np.random.default_rng(90)
    case = _rand_case(rng, 2, 3, 3, 4, T=8)
    prev = _rand_case(rng, 2, 3, 3, 4, T=2)
    cache = (prev["k"], prev["v"], prev["gamma"])
    cfg = Cfg(depth=2, C=4, c=3)
    y, W, S, _ = _run_oracle(cfg, case, cache=cache)
    yb, Wb, Sb = bf.forward(2, 4, 3, 1, 0, case["k"], case["q"], case["v"], case["theta"], case["eta"],
                            case["alpha"], case["gamma"], case["W0"], case["S0"], prev=cache)
    np.testing.assert_allclose(y, yb, rtol=1e-11, atol=1e-12)


# ---- pre-update read-out (titans-pytorch-mlx README, MAC, Eq. 21:
# h_t = M*_{t-1}(q_t)); the default reads the post-update state
# (atlas-torch README, "Known deviations from the paper's MAC")

PRE_CASES = [
    (1, 4, 1, 1, 0, 0, 3, 2, 0, 9),       # linear delta rule, several chunks
    (2, 3, 2, 1, 0, 0, 3, 3, 4, 8),       # MLP, Omega window 2
    (2, 4, 3, 1, 0, 5, 4, 4, 6, 10),      # Omega + Muon
    (1, 3, 5, 2, 0, 0, 2, 2, 0, 9),       # polynomial features, window longer than a chunk
]


@pytest.mark.parametrize("case_def", PRE_CASES)
def test_pre_update_readout_matches_bruteforce(case_def):
    depth, C, c, p, proj, ns, d_k, d_v, hidden, T = case_def
    rng = np.random.default_rng(sum(case_def) * 7919 + 1)
    case = _rand_case(rng, depth, d_k, d_v, hidden, T, p=p, proj=proj)
    y, W, S, _ = _run_oracle(Cfg(depth=depth, C=C, c=c, p=p, ns_iters=ns, readout="pre"), case)
    yb, Wb, Sb = bf.forward(depth, C, c, p, ns, case["k"], case["q"], case["v"], case["theta"], case["eta"],
                            case["alpha"], case["gamma"], case["W0"], case["S0"], case["P"], pre=True)
    np.testing.assert_allclose(y, yb, rtol=1e-10, atol=1e-11)
    for a, b in zip(W + S, Wb + Sb):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


def test_pre_update_readout_changes_only_the_readout():
    """The two read-out modes write back the same state; the pre-update
    read-out of the first token is the initial memory applied to q_0, and
    the two modes' outputs differ elsewhere (the shift is real)."""
    rng = np.random.default_rng(4242)
    case = _rand_case(rng, 2, 3, 3, 5, T=8)
    y_post, W_post, S_post, _ = _run_oracle(Cfg(depth=2, C=4, c=2), case)
    y_pre, W_pre, S_pre, _ = _run_oracle(Cfg(depth=2, C=4, c=2, readout="pre"), case)
    for a, b in zip(W_post + S_post, W_pre + S_pre):
        np.testing.assert_array_equal(a, b)
    np.testing.assert_allclose(y_pre[0], bf.apply_mem(case["W0"], case["q"][0], 2), rtol=1e-13, atol=1e-14)
    assert np.abs(y_pre[1:] - y_post[1:]).max() > 1e-6


# ---- Newton-Schulz on the windowed surprise (atlas-torch README, "Atlas
# Extensions": orthogonalisation of the surprise updates; per-token store
# path with eta outside Newton-Schulz)

SURPRISE_CASES = [
    (1, 4, 3, 1, 0, 5, 3, 2, 0, 9),       # linear memory, Omega window 3
    (2, 3, 2, 1, 0, 5, 3, 3, 4, 8),       # MLP, window 2
    (2, 4, 1, 1, 0, 3, 4, 4, 6, 8),       # MLP, c = 1 (rank-one surprise)
    (1, 3, 5, 2, 0, 5, 2, 2, 0, 9),       # polynomial features, window longer than a chunk
]


@pytest.mark.parametrize("case_def", SURPRISE_CASES)
def test_surprise_ns_matches_bruteforce(case_def):
    depth, C, c, p, proj, ns, d_k, d_v, hidden, T = case_def
    rng = np.random.default_rng(sum(case_def) * 104729 + 3)
    case = _rand_case(rng, depth, d_k, d_v, hidden, T, p=p, proj=proj)
    y, W, S, _ = _run_oracle(Cfg(depth=depth, C=C, c=c, p=p, ns_iters=ns, ns_target="surprise"), case)
    yb, Wb, Sb = bf.forward(depth, C, c, p, ns, case["k"], case["q"], case["v"], case["theta"], case["eta"],
                            case["alpha"], case["gamma"], case["W0"], case["S0"], case["P"], surprise_ns=True)
    np.testing.assert_allclose(y, yb, rtol=1e-9, atol=1e-11)
    for a, b in zip(W + S, Wb + Sb):
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-11)


def test_surprise_ns_rank_one_closed_form():
    """c = 1, linear memory, one token: the surprise 2 x^T (x W - v) is rank
    one, so NS maps it to f5(s) x_hat e_hat^T with s = |g| / (|g| + eps) and
    f5 the quintic applied five times (Muon's polynomial); the momentum and
    step size stay outside: S = eta S0 - theta f5(s) x_hat e_hat^T."""
    rng = np.random.default_rng(77)
    x = rng.standard_normal(3); q = rng.standard_normal(3); v = rng.standard_normal(2)
    W0 = 0.3 * rng.standard_normal((3, 2)); S0 = 0.1 * rng.standard_normal((3, 2))
    th, et, al = 0.07, 0.6, 0.05
    e = x @ W0 - v
    g = 2.0 * np.outer(x, e)
    s = np.linalg.norm(g) / (np.linalg.norm(g) + 1e-7)
    for _ in range(5):
        s = 3.4445 * s - 4.7750 * s ** 3 + 2.0315 * s ** 5
    S_exp = et * S0 - th * s * np.outer(x / np.linalg.norm(x), e / np.linalg.norm(e))
    W_exp = (1 - al) * W0 + S_exp
    y, W, S, _ = oracle.forward_unit(Cfg(depth=1, C=1, c=1, ns_iters=5, ns_target="surprise"), x[None], q[None],
                                     v[None], [th], [et], [al], None, [W0], [S0])
    np.testing.assert_allclose(S[0], S_exp, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(W[0], W_exp, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y[0], q @ W_exp, rtol=1e-12, atol=1e-14)


# ---- chunk-wise store path (atlas-torch README, "Bug Fixes": the
# per_token_updates flag; the titans-pytorch chunk-wise path: one summed
# gradient per chunk, pooled gates, a per-chunk scan and read-out)

CHUNKWISE_CASES = [
    # depth, C, p, proj, ns, d_k, d_v, hidden, T, readout
    (1, 4, 1, 0, 0, 4, 3, 0, 10, "post"),    # partial last chunk
    (2, 3, 1, 0, 0, 3, 3, 5, 9, "post"),
    (2, 4, 1, 0, 0, 4, 4, 6, 8, "pre"),
    (1, 3, 2, 0, 0, 2, 2, 0, 9, "post"),     # polynomial features
    (2, 4, 1, 0, 5, 4, 4, 6, 10, "post"),    # Muon on the momentum
    (2, 3, 2, 4, 3, 3, 4, 5, 9, "pre"),      # polynomial + projection + Muon
]


@pytest.mark.parametrize("case_def", CHUNKWISE_CASES)
def test_chunkwise_matches_bruteforce(case_def):
    depth, C, p, proj, ns, d_k, d_v, hidden, T, ro = case_def
    rng = np.random.default_rng(sum(x for x in case_def if isinstance(x, int)) * 31337 + len(ro))
    case = _rand_case(rng, depth, d_k, d_v, hidden, T, p=p, proj=proj)
    y, W, S, _ = _run_oracle(Cfg(depth=depth, C=C, c=1, p=p, ns_iters=ns, readout=ro, update="chunkwise"), case)
    yb, Wb, Sb = bf.forward(depth, C, 1, p, ns, case["k"], case["q"], case["v"], case["theta"], case["eta"],
                            case["alpha"], case["gamma"], case["W0"], case["S0"], case["P"], pre=(ro == "pre"),
                            chunkwise=True)
    np.testing.assert_allclose(y, yb, rtol=1e-9, atol=1e-11)
    for a, b in zip(W + S, Wb + Sb):
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("depth,ns,ro", [(1, 0, "post"), (2, 0, "post"), (2, 0, "pre"), (2, 3, "post"),
                                         (1, 5, "pre")])
def test_chunkwise_with_chunks_of_one_is_the_per_token_rule(depth, ns, ro):
    """With C = 1 a chunk is a token: pooling is the identity, the summed
    gradient is the token's own, and the chunk-end memory is W_t, so the
    chunk-wise path must give the per-token rule with c = 1 exactly."""
    rng = np.random.default_rng(500 + 10 * depth + ns)
    case = _rand_case(rng, depth, 3, 3, 4, T=7)
    a = _run_oracle(Cfg(depth=depth, C=1, c=1, ns_iters=ns, readout=ro, update="chunkwise"), case)
    b = _run_oracle(Cfg(depth=depth, C=1, c=1, ns_iters=ns, readout=ro), case)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-14)
    for x, z in zip(a[1] + a[2], b[1] + b[2]):
        np.testing.assert_allclose(x, z, rtol=1e-12, atol=1e-14)


def test_chunkwise_closed_form_one_chunk():
    """Linear memory, one chunk, eta = alpha = 0: S = -sum_t theta_t gamma_t
    2 x_t^T (x_t W0 - v_t), W = W0 + S; every token but the last reads W0,
    the last reads W."""
    rng = np.random.default_rng(606)
    T = 6
    case = _rand_case(rng, 1, 4, 3, 0, T=T)
    case["eta"] = np.zeros(T)
    case["alpha"] = np.zeros(T)
    case["S0"] = [0.2 * rng.standard_normal((4, 3))]      # eta = 0 forgets it
    y, W, S, _ = _run_oracle(Cfg(depth=1, C=T, c=1, update="chunkwise"), case)
    W0 = case["W0"][0]
    G = sum(case["theta"][t] * case["gamma"][t] * 2.0 * np.outer(case["k"][t], case["k"][t] @ W0 - case["v"][t])
            for t in range(T))
    np.testing.assert_allclose(S[0], -G, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(W[0], W0 - G, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y[:-1], case["q"][:-1] @ W0, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y[-1], case["q"][-1] @ (W0 - G), rtol=1e-12, atol=1e-14)


def test_chunkwise_gates_enter_only_through_their_chunk_mean():
    """Replacing eta and alpha by their per-chunk means changes nothing on
    the chunk-wise path, and does change the per-token rule (the pin has
    something to catch); permuting the tokens inside every chunk, last token
    kept, leaves the chunk-end memory and the outputs alike unchanged."""
    rng = np.random.default_rng(707)
    T, C = 12, 4
    case = _rand_case(rng, 2, 3, 3, 5, T=T)
    pooled = dict(case)
    for key in ("eta", "alpha"):
        pooled[key] = np.repeat(case[key].reshape(-1, C).mean(axis=1), C)
    cw = Cfg(depth=2, C=C, c=1, ns_iters=2, update="chunkwise")
    a, b = _run_oracle(cw, case), _run_oracle(cw, pooled)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-14)
    for x, z in zip(a[1] + a[2], b[1] + b[2]):
        np.testing.assert_allclose(x, z, rtol=1e-12, atol=1e-14)
    pt = Cfg(depth=2, C=C, c=1, ns_iters=2)
    assert np.abs(_run_oracle(pt, case)[1][0] - _run_oracle(pt, pooled)[1][0]).max() > 1e-6
    perm = np.concatenate([s + np.r_[rng.permutation(C - 1), C - 1] for s in range(0, T, C)])
    shuffled = {k: (v[perm] if isinstance(v, np.ndarray) and v.shape[:1] == (T,) else v) for k, v in case.items()}
    c_ = _run_oracle(cw, shuffled)
    np.testing.assert_allclose(c_[0], a[0][perm], rtol=1e-11, atol=1e-13)
    for x, z in zip(c_[1] + c_[2], a[1] + a[2]):
        np.testing.assert_allclose(x, z, rtol=1e-11, atol=1e-13)


def test_chunkwise_split_continuation():
    """Carrying the state across calls cut at a chunk edge gives the
    whole-sequence result on the chunk-wise path too."""
    rng = np.random.default_rng(808)
    T, T1, C = 16, 8, 4
    case = _rand_case(rng, 2, 4, 4, 6, T=T)
    cfg = Cfg(depth=2, C=C, c=1, ns_iters=3, update="chunkwise")
    y, W, S, _ = _run_oracle(cfg, case)
    first = {k: (v[:T1] if isinstance(v, np.ndarray) and v.shape[:1] == (T,) else v) for k, v in case.items()}
    y1, W1, S1, _ = _run_oracle(cfg, first)
    second = {k: (v[T1:] if isinstance(v, np.ndarray) and v.shape[:1] == (T,) else v) for k, v in case.items()}
    second["W0"], second["S0"] = W1, S1
    y2, W2, S2, _ = _run_oracle(cfg, second)
    np.testing.assert_allclose(np.concatenate([y1, y2]), y, rtol=1e-12, atol=1e-12)
    for a, b in zip(W2 + S2, W + S):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_chunkwise_rejects_a_window_and_surprise_ns():
    rng = np.random.default_rng(909)
    case = _rand_case(rng, 1, 3, 3, 0, T=4)
    with pytest.raises(ValueError):
        _run_oracle(Cfg(depth=1, C=2, c=2, update="chunkwise"), case)
    with pytest.raises(ValueError):
        _run_oracle(Cfg(depth=1, C=2, c=1, ns_iters=3, ns_target="surprise", update="chunkwise"), case)
