"""Why the tensor-core Newton-Schulz multiplies split bf16 pairs.  On the CPU,
five quintic steps are emulated with every product's operands rounded to
bf16 (plain), or split into a bf16 high part and a bf16 low part with three
products (hi hi + hi lo + lo hi, as the kernels issue them), accumulated in
fp64, and compared with the oracle's fp64 Newton-Schulz.  The quintic's slope
near zero (3.4445 per step) amplifies operand rounding in the small
singular directions of a momentum-like matrix: plain bf16 operands use up the
whole 2e-2 bf16 tolerance in a single call, split operands stay near 1e-4."""
import numpy as np

import oracle
from harness import bf16_round


def _bf(x):
    return bf16_round(x).astype(np.float64)


def _mm(A, B, split):
    if not split:
        return _bf(A) @ _bf(B)
    Ah, Bh = _bf(A), _bf(B)
    Al, Bl = _bf(A - Ah), _bf(B - Bh)
    return Ah @ Bh + Ah @ Bl + Al @ Bh


def _ns_emulated(G, steps, split):
    a, b, c = oracle.NS_COEFFS
    X = G / (np.linalg.norm(G) + oracle.NS_EPS)
    for _ in range(steps):
        A = _mm(X, X.T, split)
        X = a * X + _mm(b * A + c * _mm(A, A, split), X, split)
    return X


def test_split_bf16_operands_keep_newton_schulz_inside_the_tolerance():
    rng = np.random.default_rng(5)
    U, _ = np.linalg.qr(rng.standard_normal((64, 64)))
    V, _ = np.linalg.qr(rng.standard_normal((256, 64)))
    G = (U * np.geomspace(1.0, 1e-2, 64)) @ V.T       # singular values spread over two decades
    ref = oracle.newton_schulz(G, 5)

    def err(split):
        return np.abs(_ns_emulated(G, 5, split) - ref).max() / np.abs(ref).max()

    assert err(False) > 1e-2          # plain bf16: no headroom under 2e-2 after one call
    assert err(True) < 2e-4           # split bf16: two orders of magnitude of headroom
