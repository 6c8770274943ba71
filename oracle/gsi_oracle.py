"""Float64 CPU oracle for the gated linear map (TEST INFRASTRUCTURE ONLY).

This module is the parity reference for the CUDA library.  Only the test
suite, the package's smoke check and the benchmark's CPU-baseline leg may
import it; the product path never calls it and has no CPU fallback.

It follows "Gated Subspace Inference for Transformer Acceleration"
(gist.science technical summary), step by step, in the pages' notation:

  §2.1 (core decomposition):   x = V_k V_k^T x + r,   y = (W V_k)(V_k^T x) + W r = M g + W r,
                               M = W V_k (cached image), g = V_k^T x (projection).
  §2.2 (gated residual step):  rho_t = ||r|| / ||x||;  rho_t < eps -> fast path y ~= M g;
                               rho_t >= eps -> slow path, exact y = W x.
  §2.2 (Theorem 4, bound only): fast-path error per token <= ||W||_2 * eps * ||x||.

Arrays are token-major: X is T x d (row t is token x_t), W is d_out x d,
V is d x k, M is d_out x k, Y is T x d_out.  Everything is numpy float64,
computed from the stored (fp32 / bf16) values widened exactly.

Readings where the pages leave a step open (each one is listed with its
justification in the design notes):
  * tie rho == eps goes to the slow path (the pages write ">=" for slow);
  * ||x|| == 0 defines rho := 0 (fast, and M*0 = 0 = W*0);
  * a non-finite token gives rho = NaN, which is "not < eps", hence slow;
  * the residual is the explicit x - V_k g of the decomposition, never an
    identity that assumes V_k exactly orthonormal.

Pins: every function here is checked by tests that do not re-type its
formula (hand-derived examples, closed forms, invariants, brute force,
the Theorem 4 bound).  Parity of figures printed on the pages: unpinned
(the pages print no worked example).
"""
from __future__ import annotations

import numpy as np


def image(W: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Low-rank weight image M = W V_k (§2.1), d_out x k."""
    return W @ V


def gram(V: np.ndarray) -> np.ndarray:
    """Gram matrix V_k^T V_k (k x k); the identity when V_k is exactly orthonormal.

    Not a step of the method itself: the library caches it next to M so that
    it can evaluate ||x - V_k g|| without a second pass over V_k; the oracle
    provides it to check that cached artefact.
    """
    return V.T @ V


def project(X: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Subspace projection g_t = V_k^T x_t (§2.1); row t of the result is g_t."""
    return X @ V


def residual(X: np.ndarray, V: np.ndarray, G: np.ndarray) -> np.ndarray:
    """Residual r_t = x_t - V_k g_t of the exact decomposition (§2.1)."""
    return X - G @ V.T


def residual_ratio(X: np.ndarray, R: np.ndarray) -> np.ndarray:
    """rho_t = ||r_t|| / ||x_t|| (§2.2); rho := 0 for a zero token."""
    nx = np.sqrt(np.sum(X * X, axis=1))
    nr = np.sqrt(np.sum(R * R, axis=1))
    zero = nx == 0.0
    with np.errstate(invalid="ignore", divide="ignore"):
        rho = nr / np.where(zero, 1.0, nx)
    rho[zero] = 0.0
    return rho


def gate(rho: np.ndarray, eps: float) -> np.ndarray:
    """Per-token gate (§2.2): True = slow path (rho >= eps, or rho is NaN)."""
    return ~(rho < eps)


def fast_path(M: np.ndarray, G: np.ndarray) -> np.ndarray:
    """Fast path y_t ~= M g_t for every token (§2.2); rows are tokens."""
    return G @ M.T


def slow_path(W: np.ndarray, X: np.ndarray) -> np.ndarray:
    """Slow path y_t = W x_t for every token (§2.2): the dense map."""
    return X @ W.T


def compact(flags: np.ndarray):
    """Stable (ascending token index) lists of fast and slow tokens."""
    t = np.arange(len(flags), dtype=np.int64)
    return t[~flags], t[flags]


def gsi_linear(W, M, V, X, eps):
    """One gated linear map over T tokens (§2.1-§2.2).

    Returns (Y, flags, rho, G): Y is T x d_out, flags a bool array
    (True = slow), rho the residual ratios, G the projections.
    M is whatever image the caller holds (the oracle does not rebuild it).
    """
    G = project(X, V)
    R = residual(X, V, G)
    rho = residual_ratio(X, R)
    flags = gate(rho, eps)
    fast, slow = compact(flags)
    Y = np.zeros((X.shape[0], W.shape[0]))
    if len(fast):
        Y[fast] = fast_path(M, G[fast])
    if len(slow):
        Y[slow] = slow_path(W, X[slow])
    return Y, flags, rho, G


def candidates(W, M, V, X):
    """Both path results for every token: (M g_t, W x_t) rows.

    Used for tokens whose rho sits in the tolerance band around eps, where
    either gate decision is acceptable and the output must match the
    candidate of the decision actually taken.
    """
    G = project(X, V)
    return fast_path(M, G), slow_path(W, X)


def gsi_stack(maps, Xs, eps):
    """The gated map applied to a list of maps, each with its own tokens.

    maps: list of (W, M, V); Xs: list of T x d_i token blocks.  The maps are
    independent (one output per map), as in a layer's QKV / output / MLP-up /
    MLP-down projections fed with their own activations.
    """
    return [gsi_linear(W, M, V, X, eps) for (W, M, V), X in zip(maps, Xs)]


def path_errors(W, M, V, X):
    """Per-token accounting of what the fast path would cost (§2.2 and the
    Theorem 4 bound; §4's static-projection control).

    Returns (rho, err, ynorm): rho_t the residual ratio, err_t = ||M g_t - W x_t||
    (the output error token t takes on the fast path) and ynorm_t = ||W x_t||
    (the dense output's norm).
    """
    G = project(X, V)
    rho = residual_ratio(X, residual(X, V, G))
    Yf = fast_path(M, G)
    Ys = slow_path(W, X)
    return rho, np.linalg.norm(Yf - Ys, axis=1), np.linalg.norm(Ys, axis=1)


def eps_sweep(rho, err, ynorm, eps_list, tokens_per_call=1):
    """The gate at each threshold of `eps_list` (§2.2), given `path_errors`.

    For each eps: (n_slow, n_slow_calls, rel_err) with n_slow the tokens the
    gate sends to the slow path, n_slow_calls the calls (consecutive blocks
    of `tokens_per_call` tokens) that hold at least one slow token and so read
    W, and rel_err = sqrt(sum of err_t^2 over fast tokens) / sqrt(sum of
    ynorm_t^2), the gated map's relative output error against dense W x
    (slow tokens are exact).  eps = inf is the static projection: every token
    with a finite ratio takes the fast path.
    """
    rho = np.asarray(rho, dtype=np.float64)
    err = np.asarray(err, dtype=np.float64)
    y2 = float(np.sum(np.asarray(ynorm, dtype=np.float64) ** 2))
    T = len(rho)
    out = []
    for eps in eps_list:
        slow = gate(rho, eps)
        calls = [bool(slow[c:c + tokens_per_call].any()) for c in range(0, T, tokens_per_call)]
        e2 = float(np.sum(err[~slow] ** 2))
        out.append((int(slow.sum()), int(sum(calls)), float(np.sqrt(e2 / y2)) if y2 > 0 else 0.0))
    return out


def effective_params(shapes, slow_fraction):
    """Parameters a token reads on average through maps of the given
    (d, d_out, k) shapes when a fraction `slow_fraction` of its calls take
    the slow path (§4 "effective parameter count": the parameters of the
    directions the token visits): (1 - f) d_out k on the fast path (the
    image M) plus f d_out d on the slow path (W)."""
    f = float(slow_fraction)
    return float(sum((1.0 - f) * d_out * k + f * d_out * d for d, d_out, k in shapes))


# ---------------------------------------------------------------- basis construction
# "Gated Subspace Inference for Transformer Acceleration", §2.3 depth cascade
# and calibration: the basis of a layer is computed once from a calibration
# pass (the principal subspace of its activations); the next layer's basis
# starts from this one and is corrected by rank-1 updates kept orthogonal by
# DGKS re-orthogonalisation instead of a full SVD.  Readings: the principal
# subspace is the top-k eigenvectors of X^T X for a calibration block X
# (T x d); the correction is subspace iteration warm-started from the previous
# layer's basis, each step orthonormalised column by column (one rank-1 update
# of the projector per column) by classical Gram-Schmidt with the
# Daniel-Gragg-Kaufman-Stewart test: project again when the norm after a
# projection falls below eta = 1/sqrt(2) of the norm before it.


def calibration_basis(X: np.ndarray, k: int) -> np.ndarray:
    """Top-k principal directions of the activation block X (T x d): the
    eigenvectors of X^T X with the k largest eigenvalues, as the columns of a
    d x k matrix (largest first; each column's largest-magnitude entry
    positive)."""
    w, U = np.linalg.eigh(X.T @ X)
    V = U[:, np.argsort(w)[::-1][:k]]
    piv = np.argmax(np.abs(V), axis=0)
    return V * np.sign(V[piv, np.arange(V.shape[1])])[None, :]


def dgks_orthonormalize(A: np.ndarray, eta: float = 1.0 / np.sqrt(2.0)):
    """Orthonormalise the columns of A (d x k) in order by classical
    Gram-Schmidt with DGKS re-orthogonalisation.

    Column j: v = a_j; h = Q_{<j}^T v; v <- v - Q_{<j} h; if ||v|| < eta * ||a_j||
    the projection is repeated once on the result; q_j = v / ||v||.  Returns
    (Q, n_reorth), n_reorth the number of columns projected twice.
    """
    d, k = A.shape
    Q = np.zeros((d, k))
    n_reorth = 0
    for j in range(k):
        v = A[:, j].astype(np.float64).copy()
        before = np.linalg.norm(v)
        v = v - Q[:, :j] @ (Q[:, :j].T @ v)
        if np.linalg.norm(v) < eta * before:
            v = v - Q[:, :j] @ (Q[:, :j].T @ v)
            n_reorth += 1
        Q[:, j] = v / np.linalg.norm(v)
    return Q, n_reorth


def subspace_step(X: np.ndarray, V: np.ndarray):
    """One correction step: V <- DGKS-orthonormalise((X^T X) V), formed as
    X^T (X V).  Returns (V_next, n_reorth)."""
    return dgks_orthonormalize(X.T @ (X @ V))


def coherence(Va: np.ndarray, Vb: np.ndarray) -> float:
    """Mean squared cosine of the principal angles between span(Va) and
    span(Vb) (orthonormal d x k bases): ||Va^T Vb||_F^2 / k.  It is a lower
    bound on the mean cosine (each cosine lies in [0, 1])."""
    return float(np.sum((Va.T @ Vb) ** 2) / Va.shape[1])


def principal_cosines(Va: np.ndarray, Vb: np.ndarray) -> np.ndarray:
    """Cosines of the principal angles between span(Va) and span(Vb):
    the singular values of Va^T Vb, largest first."""
    return np.linalg.svd(Va.T @ Vb, compute_uv=False)


def spectral_norm(W: np.ndarray, iters: int = 200) -> float:
    """||W||_2 for the Theorem 4 bound: SVD for small W, power iteration on W^T W otherwise."""
    if W.size <= 4_000_000:
        return float(np.linalg.norm(W, 2))
    v = np.random.default_rng(0).standard_normal(W.shape[1])
    for _ in range(iters):
        v = W.T @ (W @ v)
        v /= np.linalg.norm(v)
    return float(np.linalg.norm(W @ v))


def brute_linear(W, M, V, X, eps):
    """Pure-Python loops for tiny inputs: the same steps, no BLAS.

    Serves as an independent restatement for cross-checking `gsi_linear`
    on inputs of a few dozen elements.
    """
    T, d = len(X), len(X[0])
    d_out, k = len(W), len(V[0])
    Y = [[0.0] * d_out for _ in range(T)]
    flags, rhos = [], []
    for t in range(T):
        x = [float(v) for v in X[t]]
        g = [sum(V[i][j] * x[i] for i in range(d)) for j in range(k)]
        r = [x[i] - sum(V[i][j] * g[j] for j in range(k)) for i in range(d)]
        nx = sum(v * v for v in x) ** 0.5
        nr = sum(v * v for v in r) ** 0.5
        rho = 0.0 if nx == 0.0 else nr / nx
        slow = not (rho < eps)
        for o in range(d_out):
            if slow:
                Y[t][o] = sum(W[o][i] * x[i] for i in range(d))
            else:
                Y[t][o] = sum(M[o][j] * g[j] for j in range(k))
        flags.append(slow)
        rhos.append(rho)
    return np.array(Y), np.array(flags), np.array(rhos)


def brute_image(W, V):
    """Pure-Python triple loop for M = W V_k on tiny inputs."""
    d_out, d, k = len(W), len(V), len(V[0])
    return np.array([[sum(W[o][i] * V[i][j] for i in range(d)) for j in range(k)]
                     for o in range(d_out)])
