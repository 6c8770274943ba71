"""Pins for the float64 oracle: checks against facts that do not come from it.

Each `pin_*` takes an oracle module `o` (the real one, or a copy with a
planted mistake) and raises if `o` disagrees with what the pages and the
mathematics fix:

* hand-derived closed-form examples (tests/golden/hand_examples.json);
* the decomposition's geometry (the residual is orthogonal to span(V_k) and
  is the closest point; Pythagoras for an orthonormal basis);
* special cases with closed forms (axis basis, eps = 0, eps = inf,
  x inside span(V_k), k = d);
* the Theorem 4 fast-path error bound;
* invariances (scaling by powers of two, token permutation);
* pure-Python brute force on tiny inputs.

Definitions: "Gated Subspace Inference for Transformer Acceleration"
(gist.science technical summary), §2.1 core decomposition and §2.2 gated
residual step with its Theorem 4 bound.
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _rand_basis(rs, d, k):
    q, r = np.linalg.qr(rs.standard_normal((d, k)))
    return q * np.sign(np.diag(r))[None, :]


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, f"{what}: max abs error {err} > {tol}"


def pin_hand_examples(o):
    """Every quantity of the hand-worked examples (§2.1, §2.2)."""
    ex = json.load(open(GOLDEN))["examples"]
    for e in ex:
        V = np.array(e["V"], float)
        W = np.array(e["W"], float)
        M = np.array(e["M"], float)
        tol = max(e["tol"], 1e-12)
        _close(o.image(W, V), M, tol, e["name"] + " image")
        X = np.array([t["x"] for t in e["tokens"]], float)
        G = o.project(X, V)
        _close(G, [t["g"] for t in e["tokens"]], tol, e["name"] + " g")
        R = o.residual(X, V, G)
        _close(R, [t["r"] for t in e["tokens"]], tol, e["name"] + " r")
        rho = o.residual_ratio(X, R)
        _close(rho, [t["rho"] for t in e["tokens"]], tol, e["name"] + " rho")
        flags = o.gate(rho, e["eps"])
        assert list(flags) == [t["slow"] for t in e["tokens"]], e["name"] + " flags"
        Y, f2, rho2, _ = o.gsi_linear(W, M, V, X, e["eps"])
        assert list(f2) == [t["slow"] for t in e["tokens"]], e["name"] + " flags (linear)"
        _close(Y, [t["y"] for t in e["tokens"]], tol * 100, e["name"] + " y")
        Yf, Ys = o.candidates(W, M, V, X)
        for i, t in enumerate(e["tokens"]):
            cand = Ys[i] if t["slow"] else Yf[i]
            _close(cand, t["y"], tol * 100, e["name"] + " candidate")
            if "fast_error_norm" in t:
                err = np.linalg.norm(Ys[i] - Yf[i])
                _close(err, t["fast_error_norm"], 1e-9, e["name"] + " fast error")
        if "W_spectral_norm" in e:
            _close(o.spectral_norm(W), e["W_spectral_norm"], 1e-9, e["name"] + " ||W||_2")
        # brute force restatement agrees on the same examples
        Yb, fb, rb = o.brute_linear(W.tolist(), M.tolist(), V.tolist(), X.tolist(), e["eps"])
        assert list(fb) == [t["slow"] for t in e["tokens"]], e["name"] + " brute flags"
        _close(Yb, [t["y"] for t in e["tokens"]], tol * 100, e["name"] + " brute y")


def pin_decomposition_geometry(o, seed=11):
    """r is orthogonal to span(V_k), is the closest point, and ||x||^2 = ||g||^2 + ||r||^2."""
    rs = np.random.default_rng(seed)
    d, k, T = 40, 7, 9
    V = _rand_basis(rs, d, k)
    X = rs.standard_normal((T, d))
    G = o.project(X, V)
    R = o.residual(X, V, G)
    _close(R @ V, np.zeros((T, k)), 1e-12, "V^T r")
    _close(np.sum(X * X, 1), np.sum(G * G, 1) + np.sum(R * R, 1), 1e-10, "Pythagoras")
    for _ in range(5):
        c = G + 0.1 * rs.standard_normal(G.shape)
        other = X - c @ V.T
        assert np.all(np.linalg.norm(other, axis=1) >= np.linalg.norm(R, axis=1) - 1e-12), \
            "residual is not the closest point"
    # a non-orthonormal basis: the residual is still x minus the span component V g
    B = V @ np.diag(np.linspace(0.5, 1.5, k))
    GB = o.project(X, B)
    _close(GB, X @ B, 1e-12, "projection with scaled basis")
    _close(o.residual(X, B, GB) + GB @ B.T, X, 1e-12, "x = V g + r with scaled basis")


def pin_axis_basis(o, seed=12):
    """V_k = I[:, :k]: g = x[:k], M = W[:, :k], rho = ||x[k:]||/||x|| exactly."""
    rs = np.random.default_rng(seed)
    d, d_out, k, T = 24, 10, 5, 13
    V = np.eye(d)[:, :k]
    W = rs.standard_normal((d_out, d))
    X = rs.standard_normal((T, d))
    M = o.image(W, V)
    _close(M, W[:, :k], 0.0, "axis image")
    G = o.project(X, V)
    _close(G, X[:, :k], 0.0, "axis g")
    rho = o.residual_ratio(X, o.residual(X, V, G))
    want = np.linalg.norm(X[:, k:], axis=1) / np.linalg.norm(X, axis=1)
    _close(rho, want, 1e-15, "axis rho")
    eps = float(np.median(want))
    Y, flags, _, _ = o.gsi_linear(W, M, V, X, eps)
    assert np.array_equal(flags, ~(want < eps)), "axis flags"
    for t in range(T):
        want_y = W @ X[t] if flags[t] else W[:, :k] @ X[t, :k]
        _close(Y[t], want_y, 1e-12, f"axis y[{t}]")


def _brute_dense(W, X):
    return np.array([[sum(W[o_, i] * X[t, i] for i in range(W.shape[1]))
                      for o_ in range(W.shape[0])] for t in range(X.shape[0])])


def pin_eps_zero(o, seed=13):
    """eps = 0: every token is slow and Y equals dense W x (brute force loops)."""
    rs = np.random.default_rng(seed)
    d, d_out, k, T = 12, 7, 3, 6
    V = _rand_basis(rs, d, k)
    W = rs.standard_normal((d_out, d))
    X = rs.standard_normal((T, d))
    X[2] = (V @ rs.standard_normal(k))  # a token inside the span is still slow at eps = 0
    Y, flags, _, _ = o.gsi_linear(W, o.image(W, V), V, X, 0.0)
    assert flags.all(), "eps=0 must send every token to the slow path"
    _close(Y, _brute_dense(W, X), 1e-12, "eps=0 dense")


def pin_in_span(o, seed=14):
    """x in span(V_k): r = 0, every token fast (eps > 0), M g = W x."""
    rs = np.random.default_rng(seed)
    d, d_out, k, T = 30, 11, 6, 8
    V = _rand_basis(rs, d, k)
    W = rs.standard_normal((d_out, d))
    A = rs.standard_normal((T, k))
    X = A @ V.T
    Y, flags, rho, G = o.gsi_linear(W, o.image(W, V), V, X, 1e-6)
    assert np.all(rho < 1e-13), "in-span rho"
    assert not flags.any(), "in-span tokens must be fast"
    _close(G, A, 1e-12, "in-span coefficients")
    _close(Y, _brute_dense(W, X), 1e-12, "in-span y")


def pin_full_rank(o, seed=15):
    """k = d (square orthogonal V): everything fast and exact."""
    rs = np.random.default_rng(seed)
    d, d_out, T = 9, 5, 7
    V = _rand_basis(rs, d, d)
    W = rs.standard_normal((d_out, d))
    X = rs.standard_normal((T, d))
    Y, flags, rho, _ = o.gsi_linear(W, o.image(W, V), V, X, 1e-8)
    assert not flags.any() and np.all(rho < 1e-13), "k=d is all-fast"
    _close(Y, _brute_dense(W, X), 1e-12, "k=d y")


def pin_theorem4(o, seed=16):
    """Theorem 4 (§2.2): fast-path error <= ||W||_2 * rho * ||x|| < ||W||_2 * eps * ||x||."""
    rs = np.random.default_rng(seed)
    d, d_out, k, T = 64, 48, 8, 200
    V = _rand_basis(rs, d, k)
    W = rs.standard_normal((d_out, d))
    s = rs.uniform(0.0, 0.6, T)
    X = rs.standard_normal((T, k)) @ V.T + s[:, None] * rs.standard_normal((T, d))
    eps = 0.3
    M = o.image(W, V)
    Y, flags, rho, G = o.gsi_linear(W, M, V, X, eps)
    w2 = float(np.sqrt(np.max(np.linalg.eigvalsh(W.T @ W))))
    _close(o.spectral_norm(W), w2, 1e-9 * w2, "spectral norm")
    fast = ~flags
    assert fast.sum() > 10 and flags.sum() > 10, "theorem-4 case needs both paths"
    err = np.linalg.norm(Y[fast] - X[fast] @ W.T, axis=1)
    nx = np.linalg.norm(X[fast], axis=1)
    assert np.all(err <= w2 * rho[fast] * nx * (1 + 1e-12) + 1e-12), "Theorem 4 (rho) bound"
    assert np.all(err < w2 * eps * nx), "Theorem 4 (eps) bound"
    _close(Y[flags], X[flags] @ W.T, 1e-12, "slow tokens exact")


def pin_eps_inf(o, seed=17):
    """eps = +inf is static projection: every token fast; 0 <= rho <= 1 for orthonormal V."""
    rs = np.random.default_rng(seed)
    d, d_out, k, T = 20, 6, 4, 15
    V = _rand_basis(rs, d, k)
    W = rs.standard_normal((d_out, d))
    X = rs.standard_normal((T, d)) * rs.uniform(0, 3, (T, 1))
    Y, flags, rho, G = o.gsi_linear(W, o.image(W, V), V, X, np.inf)
    assert not flags.any(), "eps=inf is all-fast"
    assert np.all((rho >= 0) & (rho <= 1 + 1e-15)), "rho in [0, 1]"
    # fast path output is the image of the projected token: W (V V^T x)
    _close(Y, (X @ V @ V.T) @ W.T, 1e-12, "static projection output")


def pin_scaling(o, seed=18):
    """x -> 2^j x leaves rho and flags unchanged and scales y by 2^j exactly."""
    rs = np.random.default_rng(seed)
    d, d_out, k, T = 16, 9, 4, 12
    V = _rand_basis(rs, d, k)
    W = rs.standard_normal((d_out, d))
    s = rs.uniform(0, 0.5, T)
    X = rs.standard_normal((T, k)) @ V.T + s[:, None] * rs.standard_normal((T, d))
    M = o.image(W, V)
    Y, f, rho, _ = o.gsi_linear(W, M, V, X, 0.2)
    for j in (-3, 5):
        Y2, f2, rho2, _ = o.gsi_linear(W, M, V, X * 2.0 ** j, 0.2)
        assert np.array_equal(f, f2) and np.array_equal(rho, rho2), "scale invariance of the gate"
        assert np.array_equal(Y2, Y * 2.0 ** j), "scale equivariance of y"


def pin_permutation(o, seed=19):
    """Permuting tokens permutes Y, rho and flags."""
    rs = np.random.default_rng(seed)
    d, d_out, k, T = 16, 9, 4, 12
    V = _rand_basis(rs, d, k)
    W = rs.standard_normal((d_out, d))
    s = rs.uniform(0, 0.5, T)
    X = rs.standard_normal((T, k)) @ V.T + s[:, None] * rs.standard_normal((T, d))
    M = o.image(W, V)
    Y, f, rho, _ = o.gsi_linear(W, M, V, X, 0.2)
    p = rs.permutation(T)
    Y2, f2, rho2, _ = o.gsi_linear(W, M, V, X[p], 0.2)
    assert np.array_equal(f2, f[p]), "permutation flags"
    _close(Y2, Y[p], 1e-13, "permutation y")
    _close(rho2, rho[p], 1e-15, "permutation rho")


def pin_degenerate_tokens(o, seed=20):
    """Zero token: rho = 0, fast, y = 0.  Non-finite token: slow, NaN propagates."""
    rs = np.random.default_rng(seed)
    d, d_out, k = 8, 5, 2
    V = _rand_basis(rs, d, k)
    W = rs.standard_normal((d_out, d))
    X = np.zeros((3, d))
    X[1, 3] = np.nan
    X[2] = rs.standard_normal(d)
    Y, flags, rho, _ = o.gsi_linear(W, o.image(W, V), V, X, 0.5)
    assert rho[0] == 0.0 and not flags[0] and np.all(Y[0] == 0.0), "zero token"
    assert flags[1] and np.isnan(rho[1]) and np.all(np.isnan(Y[1])), "NaN token"


def pin_compact(o, seed=21):
    """Stable ascending, disjoint, covering index lists; fast first element of the pair."""
    rs = np.random.default_rng(seed)
    for T in (0, 1, 7, 64):
        flags = rs.random(T) < 0.3
        fast, slow = o.compact(flags)
        assert np.all(np.diff(fast) > 0) and np.all(np.diff(slow) > 0), "ascending"
        assert not flags[fast].any() and flags[slow].all(), "fast/slow membership"
        assert len(fast) + len(slow) == T and set(fast) | set(slow) == set(range(T)), "cover"


def pin_gram(o, seed=22):
    """Gram of an orthonormal basis is I; of V D (diagonal D) it is D^2."""
    rs = np.random.default_rng(seed)
    V = _rand_basis(rs, 30, 6)
    _close(o.gram(V), np.eye(6), 1e-13, "gram of orthonormal V")
    D = np.diag([1.0, 2.0, 0.5, 3.0, 1.0, 0.25])
    _close(o.gram(V @ D), D @ D, 1e-12, "gram of scaled V")


def pin_brute(o, seed=23):
    """The BLAS-based path agrees with the pure-Python loops on tiny random inputs."""
    rs = np.random.default_rng(seed)
    d, d_out, k, T = 9, 6, 3, 8
    V = _rand_basis(rs, d, k)
    W = rs.standard_normal((d_out, d))
    s = rs.uniform(0, 0.8, T)
    X = rs.standard_normal((T, k)) @ V.T + s[:, None] * rs.standard_normal((T, d))
    M = o.image(W, V)
    _close(M, o.brute_image(W.tolist(), V.tolist()), 1e-12, "brute image")
    Y, f, rho, _ = o.gsi_linear(W, M, V, X, 0.3)
    Yb, fb, rb = o.brute_linear(W.tolist(), M.tolist(), V.tolist(), X.tolist(), 0.3)
    assert f.any() and (~f).any(), "brute case needs both paths"
    assert np.array_equal(f, fb), "brute flags"
    _close(rho, rb, 1e-12, "brute rho")
    _close(Y, Yb, 1e-12, "brute y")


def pin_stack(o):
    """A list of maps gives each map's own hand-derived result."""
    ex = json.load(open(GOLDEN))["examples"]
    a, b = ex[0], ex[2]
    maps, Xs = [], []
    for e in (a, b):
        maps.append((np.array(e["W"], float), np.array(e["M"], float), np.array(e["V"], float)))
        Xs.append(np.array([t["x"] for t in e["tokens"]], float))
    out = o.gsi_stack(maps, Xs, 0.55)
    # eps 0.55: example a: rho (0, 1, 0.6, 0) -> slow only token 1 and 2;
    # example b: rho (0.6, 0.8, 5/13) -> slow, slow, fast
    assert list(out[0][1]) == [False, True, True, False], "stack map 0 flags"
    assert list(out[1][1]) == [True, True, False], "stack map 1 flags"
    _close(out[0][0], [[11, 32], [34, 73], [44.5, 109], [0, 0]], 1e-12, "stack map 0 y")
    _close(out[1][0], [[4, 3, 8], [4, 3, 0], [12, 0, 24]], 1e-12, "stack map 1 y")


def pin_path_errors_axis(o, seed=24):
    """Axis basis V = I[:, :k]: the fast path drops exactly W[:, k:] x[k:]
    (closed form), and the dense output is W x."""
    rs = np.random.default_rng(seed)
    d, k, d_out, T = 12, 5, 7, 6
    V = np.eye(d)[:, :k]
    W = rs.standard_normal((d_out, d))
    X = rs.standard_normal((T, d))
    rho, err, ynorm = o.path_errors(W, W[:, :k], V, X)
    want_err = [np.sqrt(sum(sum(W[i, j] * x[j] for j in range(k, d)) ** 2 for i in range(d_out))) for x in X]
    want_y = [np.sqrt(sum(sum(W[i, j] * x[j] for j in range(d)) ** 2 for i in range(d_out))) for x in X]
    want_rho = [np.sqrt(sum(v * v for v in x[k:]) / sum(v * v for v in x)) for x in X]
    _close(err, want_err, 1e-12, "path_errors err (axis basis)")
    _close(ynorm, want_y, 1e-12, "path_errors ynorm (axis basis)")
    _close(rho, want_rho, 1e-12, "path_errors rho (axis basis)")


def pin_sweep_by_hand(o):
    """A sweep worked out by hand: ties go slow, NaN is slow at every eps,
    a call reads W when any of its tokens is slow."""
    rho = [0.0, 0.3, 0.5, float("nan"), 0.5]
    err = [1.0, 2.0, 3.0, 4.0, 5.0]
    ynorm = [1.0] * 5
    got = o.eps_sweep(rho, err, ynorm, [0.0, 0.3, 0.5, 0.6, float("inf")], tokens_per_call=2)
    want = [(5, 3, 0.0), (4, 3, np.sqrt(1 / 5)), (3, 2, 1.0), (1, 1, np.sqrt(39 / 5)), (1, 1, np.sqrt(39 / 5))]
    for g, w in zip(got, want):
        assert g[0] == w[0] and g[1] == w[1], f"sweep counts {g[:2]} != {w[:2]}"
        assert abs(g[2] - w[2]) <= 1e-12, f"sweep error {g[2]} != {w[2]}"


def pin_sweep_theorem4(o, seed=25):
    """On an orthonormal basis every token's fast-path error obeys the
    Theorem 4 bound ||W||_2 rho ||x||; the sweep is monotone in eps
    (fewer slow tokens, larger error), exact at eps = 0, and at eps = inf
    equals the static projection's error ||G M^T - X W^T|| / ||X W^T||."""
    rs = np.random.default_rng(seed)
    d, k, d_out, T = 40, 6, 9, 30
    V = _rand_basis(rs, d, k)
    W = rs.standard_normal((d_out, d))
    X = (V @ rs.standard_normal((k, T))).T + 0.3 * rs.standard_normal((T, d))
    M = W @ V
    rho, err, ynorm = o.path_errors(W, M, V, X)
    w2 = np.linalg.svd(W, compute_uv=False)[0]
    bound = w2 * rho * np.linalg.norm(X, axis=1)
    assert np.all(err <= bound * (1 + 1e-9) + 1e-12), "Theorem 4 bound violated"
    eps = [0.0, 0.05, 0.1, 0.2, 0.4, 0.8, float("inf")]
    sw = o.eps_sweep(rho, err, ynorm, eps)
    assert sw[0][0] == T and sw[0][2] == 0.0, "eps = 0: every token slow, exact"
    assert all(a[0] >= b[0] for a, b in zip(sw, sw[1:])), "slow count not monotone"
    assert all(a[2] <= b[2] + 1e-15 for a, b in zip(sw, sw[1:])), "error not monotone"
    static = np.linalg.norm((X @ V) @ M.T - X @ W.T) / np.linalg.norm(X @ W.T)
    assert sw[-1][0] == 0 and abs(sw[-1][2] - static) <= 1e-12, "eps = inf is the static projection"


def pin_effective_params(o):
    """Effective parameters: d_out k per map on the fast path, d_out d on the slow path."""
    assert o.effective_params([(4, 2, 1)], 0.0) == 2.0
    assert o.effective_params([(4, 2, 1)], 1.0) == 8.0
    assert o.effective_params([(4, 2, 1), (3, 5, 2)], 0.5) == 0.5 * (2 + 10) + 0.5 * (8 + 15)
    six_b = [(4096, 12288, 256), (4096, 4096, 256), (4096, 16384, 256), (16384, 4096, 256)]
    assert o.effective_params(six_b, 0.0) == (12288 + 4096 + 16384 + 4096) * 256


def pin_dgks_qr(o, seed=26):
    """DGKS Gram-Schmidt on a well-conditioned A is the thin QR of A with a
    positive R diagonal (the textbook factorisation, here through numpy's
    Householder QR): Q^T Q = I, and no column needs a second projection."""
    rs = np.random.default_rng(seed)
    A = rs.standard_normal((30, 6))
    Q, n = o.dgks_orthonormalize(A)
    q, r = np.linalg.qr(A)
    _close(Q, q * np.sign(np.diag(r))[None, :], 1e-12, "DGKS Q vs QR")
    assert n == 0, "a well-conditioned A needs no re-orthogonalisation"


def pin_dgks_reorth(o):
    """Hand example: the second column is almost the first; after one
    projection only 1e-9 of it is left (< ||a|| / sqrt 2), so it is projected
    again; Q is the identity."""
    A = np.array([[1.0, 1.0, 0.0], [0.0, 1e-9, 0.0], [0.0, 0.0, 5.0]])
    Q, n = o.dgks_orthonormalize(A)
    _close(Q, np.eye(3), 1e-15, "DGKS hand example Q")
    assert n == 1, f"re-orthogonalised {n} columns, want 1"


def _spectral_block(rs, T=60, d=24, r=10):
    """X = A diag(sigma) U^T with known principal directions U (distinct,
    decreasing sigma)."""
    A = _rand_basis(rs, T, r)
    U = _rand_basis(rs, d, r)
    sig = np.linspace(3.0, 0.5, r)
    return (A * sig[None, :]) @ U.T, U


def pin_calibration_basis(o, seed=27):
    """The calibration basis of X = A diag(sigma) U^T is U[:, :k] up to the
    column signs, which put each column's largest-magnitude entry positive."""
    rs = np.random.default_rng(seed)
    X, U = _spectral_block(rs)
    k = 4
    V = o.calibration_basis(X, k)
    _close(np.abs(V.T @ U[:, :k]), np.eye(k), 1e-10, "calibration basis vs U_k")
    piv = np.argmax(np.abs(V), axis=0)
    assert np.all(V[piv, np.arange(k)] > 0), "sign convention"


def pin_subspace_iteration(o, seed=28):
    """Subspace iteration reaches the principal subspace from a random start
    (gap sigma_4 / sigma_5 > 1), and the principal subspace is a fixed point."""
    rs = np.random.default_rng(seed)
    X, U = _spectral_block(rs)
    k = 4
    V = _rand_basis(rs, X.shape[1], k)
    for _ in range(80):
        V, _ = o.subspace_step(X, V)
    Uk = U[:, :k]
    assert np.sum((Uk.T @ V) ** 2) / k >= 1 - 1e-10, "did not converge to span(U_k)"
    W, _ = o.subspace_step(X, Uk)
    assert np.sum((Uk.T @ W) ** 2) / k >= 1 - 1e-13, "principal subspace not fixed"


def pin_coherence(o):
    """Hand example: lines at angle theta in the plane have cos^2 theta;
    a basis with itself 1, with its orthogonal complement 0."""
    th = 0.3
    a = np.array([[1.0], [0.0]])
    b = np.array([[np.cos(th)], [np.sin(th)]])
    assert abs(o.coherence(a, b) - np.cos(th) ** 2) <= 1e-15
    _close(o.principal_cosines(a, b), [np.cos(th)], 1e-15, "principal cosine")
    I = np.eye(4)
    assert o.coherence(I[:, :2], I[:, :2]) == 1.0 and o.coherence(I[:, :2], I[:, 2:]) == 0.0


def pin_spectral_norm_large(o, seed=29):
    """The power-iteration branch of ||W||_2 (maps above 4 M elements) against a
    closed form: W block-diagonal with 2 x 2 blocks B, whose spectral norm is
    max over blocks of sqrt((t + sqrt(t^2 - 4 det(B)^2)) / 2), t = ||B||_F^2.
    One block is scaled so its norm leads the rest by 10% (power iteration on
    W^T W then converges as 0.81 per step)."""
    rs = np.random.default_rng(seed)
    nb = 1025  # 2050 x 2050 = 4.2 M elements: the large-map branch
    B = rs.standard_normal((nb, 2, 2))
    t = np.sum(B * B, axis=(1, 2))
    det = B[:, 0, 0] * B[:, 1, 1] - B[:, 0, 1] * B[:, 1, 0]
    norms = np.sqrt((t + np.sqrt(t * t - 4.0 * det * det)) / 2.0)
    top = int(rs.integers(nb))
    rest = np.max(np.delete(norms, top))
    B[top] *= 1.1 * rest / norms[top]
    want = 1.1 * rest
    W = np.zeros((2 * nb, 2 * nb))
    for b in range(nb):
        W[2 * b:2 * b + 2, 2 * b:2 * b + 2] = B[b]
    assert W.size > 4_000_000
    _close(o.spectral_norm(W), want, 1e-9 * want, "spectral norm, power-iteration branch")


ALL_PINS = [
    pin_hand_examples, pin_decomposition_geometry, pin_axis_basis, pin_eps_zero,
    pin_in_span, pin_full_rank, pin_theorem4, pin_eps_inf, pin_scaling,
    pin_permutation, pin_degenerate_tokens, pin_compact, pin_gram, pin_brute,
    pin_stack, pin_path_errors_axis, pin_sweep_by_hand, pin_sweep_theorem4, pin_effective_params,
    pin_dgks_qr, pin_dgks_reorth, pin_calibration_basis, pin_subspace_iteration, pin_coherence,
    pin_spectral_norm_large,
]
