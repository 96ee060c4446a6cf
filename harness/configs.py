"""Named workloads of the memory-layer forward, by shape.

Each workload fixes the memory (depth, widths), the chunking (C tokens per
chunk, Omega window c), the key feature map (polynomial degree p, optional
projection back to ``proj_dim``), the number of Newton-Schulz iterations, the
input precision and the batch geometry (B batches x H heads x T tokens).

Sources of the shapes: the Titans update (titans-pytorch-mlx README, "Core
Equations", Eq. 12-14), the ATLAS summary (Sections 3.1-3.3 and 5) and the
atlas-torch README ("Atlas Extensions" table).
"""
from __future__ import annotations

import dataclasses
from math import comb


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    depth: int          # 1 = matrix memory, 2 = residual SiLU MLP memory
    d_k: int            # key / query width before the feature map
    d_v: int            # value width (== memory output width)
    hidden: int         # MLP hidden width (depth 2 only, else 0)
    C: int              # tokens per chunk (weights frozen at chunk start)
    c: int              # Omega window: the last c tokens, including t
    p: int              # polynomial feature degree, 1 or 2
    proj_dim: int       # 0: no projection, else features are projected to this width
    ns_iters: int       # Newton-Schulz iterations on the momentum, 0 = off
    qkv_dtype: str      # "f32" or "bf16"
    B: int
    H: int
    T: int
    seed: int
    use_gamma: bool = False       # per-token Omega weights drawn, else all ones
    alpha_mu: float = -4.0        # mean of the normal under the decay sigmoid
    w0_init: str = "zero"         # "zero" or "xavier" (per head, shared over B)
    readout: str = "post"         # "post": y_t from the memory after token t's update; "pre": before it
    ns_target: str = "momentum"   # Newton-Schulz on the momentum, or "surprise": on each token's windowed gradient
    update: str = "per_token"     # or "chunkwise": one summed gradient, pooled gates and one step per chunk
    theta_scale: float = 0.1      # theta = theta_scale * sigmoid(N(0, 1))

    @property
    def units(self) -> int:
        return self.B * self.H

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.T

    @property
    def poly_dim(self) -> int:
        """Width of the degree-p monomial expansion of a d_k vector."""
        return self.d_k if self.p == 1 else comb(self.d_k + 2, 2)

    @property
    def feat_dim(self) -> int:
        """Width of the memory input after feature map and projection."""
        return self.proj_dim if self.proj_dim else self.poly_dim

    def matrix_shapes(self):
        """Shapes of the memory weight matrices (row-vector convention)."""
        if self.depth == 1:
            return [(self.feat_dim, self.d_v)]
        return [(self.feat_dim, self.hidden), (self.hidden, self.d_v)]

    def scaled(self, **kw) -> "Workload":
        """Same method settings, different geometry (for small parity cases)."""
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # Linear memory, all fp32, one head.
    "linear_f32": Workload(
        "linear_f32", depth=1, d_k=32, d_v=32, hidden=0, C=16, c=1, p=1,
        proj_dim=0, ns_iters=0, qkv_dtype="f32", B=1, H=1, T=256, seed=0),
    # Titans memory: 2-layer residual SiLU MLP 64 -> 256 -> 64.
    "titans_mlp": Workload(
        "titans_mlp", depth=2, d_k=64, d_v=64, hidden=256, C=64, c=1, p=1,
        proj_dim=0, ns_iters=0, qkv_dtype="bf16", B=4, H=8, T=4096, seed=1,
        w0_init="xavier"),
    # ATLAS Omega rule on degree-2 features of 32-dim keys (561 features).
    "atlas_poly_c4": Workload(
        "atlas_poly_c4", depth=1, d_k=32, d_v=64, hidden=0, C=64, c=4, p=2,
        proj_dim=0, ns_iters=0, qkv_dtype="bf16", B=2, H=8, T=8192, seed=2,
        use_gamma=True),
    "atlas_poly_c16": Workload(
        "atlas_poly_c16", depth=1, d_k=32, d_v=64, hidden=0, C=64, c=16, p=2,
        proj_dim=0, ns_iters=0, qkv_dtype="bf16", B=2, H=8, T=8192, seed=2,
        use_gamma=True),
    # ATLAS with Muon: 128 -> 512 -> 128 MLP, window 8, 5 NS iterations.
    "atlas_muon": Workload(
        "atlas_muon", depth=2, d_k=128, d_v=128, hidden=512, C=64, c=8, p=1,
        proj_dim=0, ns_iters=5, qkv_dtype="bf16", B=2, H=16, T=16384, seed=3,
        w0_init="xavier"),
    # ATLAS with Newton-Schulz on the windowed surprise (eta, theta outside
    # NS) instead of the momentum; otherwise the Muon workload.
    "atlas_muon_surprise": Workload(
        "atlas_muon_surprise", depth=2, d_k=128, d_v=128, hidden=512, C=64, c=8, p=1,
        proj_dim=0, ns_iters=5, qkv_dtype="bf16", B=2, H=16, T=16384, seed=3,
        w0_init="xavier", ns_target="surprise"),
    # The chunk-wise store path of titans-pytorch (one summed gradient per
    # chunk, pooled eta / alpha, one momentum and decay step per chunk) on
    # the Titans memory, and with Muon on the Muon geometry (no Omega window
    # on that path: c = 1).  Without Muon the chunk's step is the sum of C
    # token steps, so theta is drawn C times smaller: with the per-token
    # scale this memory diverges within ~1000 tokens, in fp64 as well.
    "titans_chunkwise": Workload(
        "titans_chunkwise", depth=2, d_k=64, d_v=64, hidden=256, C=64, c=1, p=1,
        proj_dim=0, ns_iters=0, qkv_dtype="bf16", B=4, H=8, T=4096, seed=1,
        w0_init="xavier", update="chunkwise", theta_scale=0.1 / 64),
    "atlas_muon_chunkwise": Workload(
        "atlas_muon_chunkwise", depth=2, d_k=128, d_v=128, hidden=512, C=64, c=1, p=1,
        proj_dim=0, ns_iters=5, qkv_dtype="bf16", B=2, H=16, T=16384, seed=3,
        w0_init="xavier", update="chunkwise"),
    # The Titans memory with slow forgetting and a smaller step (alpha mean
    # -8, theta = 0.02 sigmoid).  With the default gates the memory decays
    # to ~1e-8 by T = 4096, so late read-outs equal the queries; here W
    # stays ~0.2 over the whole sequence, so every read-out tests the
    # memory.  (alpha mean -8 with theta 0.1 diverges, in fp64 as well.)
    "titans_mlp_slow": Workload(
        "titans_mlp_slow", depth=2, d_k=64, d_v=64, hidden=256, C=64, c=1, p=1,
        proj_dim=0, ns_iters=0, qkv_dtype="bf16", B=4, H=8, T=4096, seed=5,
        w0_init="xavier", alpha_mu=-8.0, theta_scale=0.02),
    # Long context: degree-2 features of 64-dim keys (2145) projected to 64.
    "atlas_long": Workload(
        "atlas_long", depth=2, d_k=64, d_v=64, hidden=256, C=64, c=8, p=2,
        proj_dim=64, ns_iters=5, qkv_dtype="bf16", B=1, H=16, T=131072, seed=4,
        alpha_mu=-6.0, w0_init="xavier"),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


@dataclasses.dataclass(frozen=True)
class Prologue:
    """The stage in front of the memory: x [B, T, D] -> q, k, v [B, H, T, d]
    and the gates [B, H, T] through one projection, a causal depthwise
    convolution of ``conv`` taps on the q/k/v channels, q/k L2 normalisation
    and one sigmoid head per gate and head."""
    name: str
    D: int              # model width
    H: int
    d_k: int
    d_v: int
    conv: int           # taps of the short causal convolution (4 on the pages)
    with_gamma: bool    # a fourth gate head gives the Omega weights gamma
    theta_max: float    # theta = theta_max * sigmoid(.)
    qkv_dtype: str      # type of x, W_in and the q, k, v outputs
    B: int
    T: int
    seed: int
    alpha_bias: float = -4.0   # bias of the decay head (the memory inputs' alpha mean)

    @property
    def G(self) -> int:
        return 4 if self.with_gamma else 3

    @property
    def Nc(self) -> int:
        """Convolved channels: the q, k and v heads."""
        return self.H * (2 * self.d_k + self.d_v)

    @property
    def N(self) -> int:
        """Projection width: the q/k/v channels, then G logit columns per head."""
        return self.Nc + self.G * self.H

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def scaled(self, **kw) -> "Prologue":
        return dataclasses.replace(self, **kw)


PROLOGUES = {
    # In front of the Titans memory (8 heads of 64 on a 512-wide model).
    "titans_prologue": Prologue(
        "titans_prologue", D=512, H=8, d_k=64, d_v=64, conv=4, with_gamma=False, theta_max=0.1,
        qkv_dtype="bf16", B=4, T=4096, seed=11),
    # The atlas-torch configuration example: 768 wide, 16 heads of 48,
    # with the Omega weights' gate head.
    "atlas_prologue": Prologue(
        "atlas_prologue", D=768, H=16, d_k=48, d_v=48, conv=4, with_gamma=True, theta_max=0.1,
        qkv_dtype="bf16", B=2, T=8192, seed=12),
    # fp32 throughout, odd widths.
    "small_prologue_f32": Prologue(
        "small_prologue_f32", D=40, H=3, d_k=8, d_v=12, conv=4, with_gamma=True, theta_max=0.1,
        qkv_dtype="f32", B=2, T=100, seed=13),
}
