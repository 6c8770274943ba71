"""Seeded synthetic inputs for the gated linear map.

This module only *draws* inputs: Gaussian weights, an orthonormal basis taken
from the QR factor of a Gaussian matrix, and tokens mixed from the basis plus
isotropic noise.  It holds none of the gated map's own arithmetic (no
projection, no residual ratio, no gate, no image), so both sides of a parity
check -- the float64 oracle and the CUDA library -- can consume its output
without sharing any of the method.

The pages' workloads are trained GPT-J / OPT / GPT-2 activations and weights
("Gated Subspace Inference for Transformer Acceleration", §4); none are
available here, so these synthetic stand-ins reproduce their *shapes* (the
6B and 13B projection sizes) and the low-rank-plus-noise activation structure
the method assumes (§1: activations lie near a k-dimensional subspace).

Every array is drawn in float64 from numpy's PCG64, then rounded once to the
storage dtype (round-to-nearest-even through torch).  Callers upload those
exact bytes to the device and widen the same bytes to float64 for the oracle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

# Projection shapes (d_out, d) of one decoder layer, per role.
SHAPES_6B = {
    "qkv": (12288, 4096),
    "out": (4096, 4096),
    "up": (16384, 4096),
    "down": (4096, 16384),
}
SHAPES_13B = {
    "qkv": (15360, 5120),
    "out": (5120, 5120),
    "up": (13824, 5120),
    "down": (5120, 13824),
}
ROLES = ("qkv", "out", "up", "down")
ROLE_ID = {r: i for i, r in enumerate(ROLES)}

# Purpose codes mixed into the seed so that W, V, the token draws and the
# slow-token labels of one map come from independent streams.
_W, _V, _A, _N, _LBL, _CHAIN, _FRAC, _CAL = 1, 2, 3, 4, 5, 6, 7, 8


def rng(config: int, layer: int, role: int, purpose: int) -> np.random.Generator:
    """Independent PCG64 stream for (config, layer, role, purpose)."""
    return np.random.default_rng([config, layer, role, purpose])


def storage(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    """Round a float array once to the storage dtype (RNE), as a CPU tensor."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(dtype).contiguous()


def widen(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of stored values (bf16 and fp32 widen exactly)."""
    return t.detach().cpu().to(torch.float64).numpy()


def gaussian_weight(g: np.random.Generator, d_out: int, d: int) -> np.ndarray:
    """W ~ N(0, 1/fan_in), drawn in float32 (the draw itself is not the method)."""
    w = g.standard_normal((d_out, d), dtype=np.float32)
    w *= np.float32(1.0 / math.sqrt(d))
    return w


def orthonormal_basis(g: np.random.Generator, d: int, k: int) -> np.ndarray:
    """Q factor of QR(d x k N(0,1)) in float64, signs fixed so diag(R) > 0."""
    a = g.standard_normal((d, k))
    return orth(a)


def orth(a: np.ndarray) -> np.ndarray:
    """Orthonormal basis of the columns of `a` (reduced QR, diag(R) > 0)."""
    q, r = np.linalg.qr(a, mode="reduced")
    s = np.sign(np.diag(r))
    s[s == 0] = 1.0
    return q * s[None, :]


def noise_scale(rho_target: float, d: int, k: int) -> float:
    """Noise level s giving E-residual-ratio ~= rho_target for x = V a + s n.

    With a ~ N(0, I_k), n ~ N(0, I_d): E||x||^2 = k + s^2 d and the part of
    s n outside span(V) has E-norm^2 s^2 (d - k); solving
    rho^2 = s^2 (d - k) / (k + s^2 d) for s gives the expression below.
    """
    r2 = rho_target * rho_target
    return rho_target * math.sqrt(k) / math.sqrt(d - k - r2 * d)


def mixed_tokens(g_a: np.random.Generator, g_n: np.random.Generator,
                 V: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Tokens x_t = V a_t + s_t n_t (float64, T x d)."""
    d, k = V.shape
    T = len(scales)
    a = g_a.standard_normal((T, k))
    n = g_n.standard_normal((T, d))
    return a @ V.T + scales[:, None] * n


def two_level_scales(g: np.random.Generator, T: int, n_slow: int,
                     s_fast: float, s_slow: float) -> np.ndarray:
    """Exactly n_slow tokens at s_slow, the rest at s_fast, seeded positions."""
    s = np.full(T, s_fast)
    s[g.permutation(T)[:n_slow]] = s_slow
    return s


@dataclass
class MapInputs:
    """One linear map and its tokens, in storage dtype (CPU tensors)."""
    name: str
    W: torch.Tensor          # d_out x d
    V: torch.Tensor          # d x k
    X: torch.Tensor          # T x d
    eps: float
    V64: np.ndarray = field(repr=False, default=None)  # unrounded basis (generator side only)

    @property
    def d(self):
        return self.W.shape[1]

    @property
    def d_out(self):
        return self.W.shape[0]

    @property
    def k(self):
        return self.V.shape[1]

    @property
    def T(self):
        return self.X.shape[0]


EPS = 0.05


def config1() -> MapInputs:
    """Single layer, fp32: d=256, d_out=256, k=16, T=64, eps=0.05.

    48 tokens (75%) at s=0.01 and 16 (25%) at s=0.2, seeded positions.
    """
    c, d, d_out, k, T = 1, 256, 256, 16, 64
    V64 = orthonormal_basis(rng(c, 0, 0, _V), d, k)
    W = gaussian_weight(rng(c, 0, 0, _W), d_out, d)
    s = two_level_scales(rng(c, 0, 0, _LBL), T, 16, 0.01, 0.2)
    X = mixed_tokens(rng(c, 0, 0, _A), rng(c, 0, 0, _N), V64, s)
    return MapInputs("cfg1", storage(W, torch.float32), storage(V64, torch.float32),
                     storage(X, torch.float32), EPS, V64)


def map_6b(role: str, T: int = 256, n_slow: int = 26, k: int = 256,
           layer: int = 0, config: int = 2, eps: float = EPS) -> MapInputs:
    """One 6B-class projection at bf16 with T single tokens.

    Two-level noise mixture: exactly n_slow tokens use s(4 eps), the rest
    s(eps/4), so that the slow fraction is fixed and few tokens sit near eps.
    """
    d_out, d = SHAPES_6B[role]
    m = ROLE_ID[role]
    V64 = orthonormal_basis(rng(config, layer, m, _V), d, k)
    W = gaussian_weight(rng(config, layer, m, _W), d_out, d)
    s = two_level_scales(rng(config, layer, m, _LBL), T, n_slow,
                         noise_scale(eps / 4, d, k), noise_scale(4 * eps, d, k))
    X = mixed_tokens(rng(config, layer, m, _A), rng(config, layer, m, _N), V64, s)
    return MapInputs(f"6b.{role}", storage(W, torch.bfloat16), storage(V64, torch.bfloat16),
                     storage(X, torch.bfloat16), eps, V64)


def depth_chain(config: int, role: int, d: int, k: int, n_layers: int) -> list:
    """Depth-coherent bases V^(l+1) = orth(V^(l) + 0.1 N(0,1)/sqrt(d)), float64."""
    out = [orthonormal_basis(rng(config, 0, role, _V), d, k)]
    g = rng(config, 0, role, _CHAIN)
    for _ in range(1, n_layers):
        out.append(orth(out[-1] + 0.1 * g.standard_normal((d, k)) / math.sqrt(d)))
    return out


def layer_slow_fractions(config: int, n_layers: int, lo=0.05, hi=0.15) -> np.ndarray:
    """Per-layer slow-token fraction f_l ~ U[lo, hi] (seeded)."""
    return rng(config, 0, 0, _FRAC).uniform(lo, hi, n_layers)


def map_tokens(config: int, layer: int, role: int, V64: np.ndarray, T: int, f_slow: float,
               eps: float = EPS, bernoulli: bool = False, salt: int = 0) -> torch.Tensor:
    """T bf16 tokens for one map: slow ones at s(4 eps), fast ones at s(eps/4).

    Slow tokens are either exactly round(f_slow*T) seeded positions, or
    per-token Bernoulli(f_slow) labels (exact at f=0 and f=1).  `salt`
    separates token sets drawn for the same map.
    """
    d, k = V64.shape
    gl = rng(config, layer, role, _LBL * 1000 + salt)
    s_fast, s_slow = noise_scale(eps / 4, d, k), noise_scale(4 * eps, d, k)
    if bernoulli:
        s = np.where(gl.random(T) < f_slow, s_slow, s_fast)
    else:
        s = two_level_scales(gl, T, int(round(f_slow * T)), s_fast, s_slow)
    X = mixed_tokens(rng(config, layer, role, _A * 1000 + salt),
                     rng(config, layer, role, _N * 1000 + salt), V64, s)
    return storage(X, torch.bfloat16)


def stack_layer(config: int, layer: int, basis_by_role: dict, shapes: dict,
                T: int, f_slow: float, eps: float = EPS, bernoulli: bool = False,
                roles=ROLES) -> list:
    """All maps of one layer for a stack workload (bf16): W, V and T tokens each."""
    maps = []
    for role in roles:
        m = ROLE_ID[role]
        d_out, d = shapes[role]
        V64 = basis_by_role[role]
        W = gaussian_weight(rng(config, layer, m, _W), d_out, d)
        X = map_tokens(config, layer, m, V64, T, f_slow, eps, bernoulli)
        maps.append(MapInputs(f"c{config}.l{layer}.{role}", storage(W, torch.bfloat16),
                              storage(V64, torch.bfloat16), X, eps, V64))
    return maps


def config5(T: int = 2048, n_slow: int = 410) -> MapInputs:
    """Prefill-sized map: T=2048, d=4096, d_out=16384, k=256, 410 slow tokens."""
    return map_6b("up", T=T, n_slow=n_slow, k=256, config=5)


def layer_weight_rows(config: int, layer: int, role: int, d_out: int):
    """Seeded row permutation and signs that derive layer `layer`'s W from its
    role's base Gaussian draw (W_l = S_l P_l W_base): still N(0, 1/fan_in),
    distinct per layer, and cheap to form for deep stacks."""
    g = rng(config, layer, role, _W * 1000 + 7)
    perm = g.permutation(d_out)
    signs = np.where(g.random(d_out) < 0.5, -1.0, 1.0).astype(np.float32)
    return perm, signs


def stack_config3(n_layers: int = 28, steps: int = 512, k: int = 256, eps: float = EPS):
    """28-layer linear-only stack of the 6B shapes with depth-coherent bases.

    Returns (bases, fractions, base_W, tokens): bases[role][l] float64 d x k,
    fractions[l] the layer's slow-token fraction, base_W[role] the role's
    base weight draw (bf16 tensor), tokens[(l, role)] a steps x d bf16 tensor
    of per-step activations in span(V^(l)) plus noise.
    """
    c = 3
    fr = layer_slow_fractions(c, n_layers)
    bases, base_W = {}, {}
    for role in ROLES:
        d_out, d = SHAPES_6B[role]
        r = ROLE_ID[role]
        bases[role] = depth_chain(c, r, d, k, n_layers)
        base_W[role] = storage(gaussian_weight(rng(c, 0, r, _W), d_out, d), torch.bfloat16)
    tokens = {}
    for l in range(n_layers):
        for role in ROLES:
            tokens[(l, role)] = map_tokens(c, l, ROLE_ID[role], bases[role][l], steps, float(fr[l]), eps)
    return bases, fr, base_W, tokens


def calibration_stream(config: int, n_layers: int, d: int, m: int, T: int, decay: float = 0.97,
                       noise: float = 0.01, role: int = 0, gap_at: int = 0, gap: float = 1.0):
    """Depth-coherent calibration blocks for basis construction.

    Layer l's activations are x = U^(l) diag(sigma) a + noise * n with
    U^(l) (d x m) the depth chain U^(l+1) = orth(U^(l) + 0.1 N(0,1)/sqrt(d)),
    sigma_i = decay^i (a gradual spectrum, so the principal subspace is not
    found in one step), multiplied by `gap` for i >= gap_at when gap_at > 0
    (a spectral gap that makes the top-gap_at subspace well defined),
    a ~ N(0, I_m), n ~ N(0, I_d).  Returns
    (U_list float64, blocks) with blocks[l] a T x d float64 array; round it
    to the storage dtype with `storage`.
    """
    U = depth_chain(config, role, d, m, n_layers)
    sig = decay ** np.arange(m)
    if gap_at > 0:
        sig[gap_at:] *= gap
    blocks = []
    for l in range(n_layers):
        g = rng(config, l, role, _CAL)
        a = g.standard_normal((T, m)) * sig[None, :]
        blocks.append(a @ U[l].T + noise * g.standard_normal((T, d)))
    return U, blocks


def random_basis_t(config: int, k: int, d: int, salt: int = 0) -> np.ndarray:
    """A seeded random start for basis construction: k x d Gaussian rows
    (orthonormalised by the code under test)."""
    return rng(config, 0, 0, _CAL * 1000 + salt).standard_normal((k, d))


def stack_config4(n_layers: int = 40, k: int = 320, pool: int = 64, eps: float = EPS):
    """40-layer stack of the 13B shapes at k = 320 (bf16), built cheaply.

    Per role: one base weight draw W_base ~ N(0, 1/fan_in) and one basis
    V_base; layer l's weight is a seeded row permutation with random signs of
    W_base (still N(0, 1/fan_in), distinct per layer) and its basis a seeded
    column permutation of V_base (still orthonormal, the same subspace).
    Tokens come from two pools per role drawn from V_base -- `pool` at the
    fast noise level s(eps/4) and `pool` at the slow one s(4 eps) -- so any
    layer's tokens can be picked by per-token slow labels (see pool_tokens).

    Returns (base_W, V64, layer_rows, layer_cols, pools): base_W[role] a bf16
    tensor, V64[role] float64 d x k, layer_rows[(l, role)] = (perm, signs),
    layer_cols[(l, role)] a permutation of range(k), pools[role] =
    (fast, slow) bf16 tensors of pool x d.
    """
    c = 4
    base_W, V64, rows, cols, pools = {}, {}, {}, {}, {}
    for role in ROLES:
        d_out, d = SHAPES_13B[role]
        r = ROLE_ID[role]
        base_W[role] = storage(gaussian_weight(rng(c, 0, r, _W), d_out, d), torch.bfloat16)
        V64[role] = orthonormal_basis(rng(c, 0, r, _V), d, k)
        pools[role] = (map_tokens(c, 0, r, V64[role], pool, 0.0, eps, salt=1),
                       map_tokens(c, 0, r, V64[role], pool, 1.0, eps, salt=2))
        for l in range(n_layers):
            rows[(l, role)] = layer_weight_rows(c, l, r, d_out)
            cols[(l, role)] = rng(c, l, r, _CHAIN * 1000 + 1).permutation(k)
    return base_W, V64, rows, cols, pools


def pool_tokens(pools, role: str, layer: int, n: int, f_slow: float, salt: int = 0) -> torch.Tensor:
    """n bf16 tokens for one map of the config-4 stack: per-token Bernoulli(f)
    slow labels (exact at f = 0 and f = 1), each token a seeded pick from the
    role's slow or fast pool."""
    fast, slow = pools[role]
    g = rng(4, layer, ROLE_ID[role], _LBL * 1000 + 500 + salt)
    lab = g.random(n) < f_slow
    pick = torch.from_numpy(g.integers(0, fast.shape[0], n))
    X = fast[pick].clone()
    if lab.any():
        m = torch.from_numpy(lab)
        X[m] = slow[pick[m]]
    return X.contiguous()
