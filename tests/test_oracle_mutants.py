"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that the pins catch every one of them.

Each mutant edits one line of the oracle's source text -- a flipped sign, a
dropped term, a transposed operand, a wrong comparison, a wrong index -- and
re-executes it as a separate module.  The real oracle is never modified.
"""
import inspect
import types

import pytest

from oracle import gsi_oracle
from tests.oracle_pins import ALL_PINS

SRC = inspect.getsource(gsi_oracle)

MUTANTS = {
    "image_drops_basis": ("return W @ V\n", "return W[:, :V.shape[1]]\n"),
    "image_transposed": ("return W @ V\n", "return (V.T @ W.T).T[:, ::-1]\n"),
    "project_wrong_rows": ("return X @ V\n", "return X[:, :V.shape[1]]\n"),
    "residual_sign": ("return X - G @ V.T", "return X + G @ V.T"),
    "residual_dropped": ("return X - G @ V.T", "return X"),
    "ratio_squared_norm": ("rho = nr / np.where(zero, 1.0, nx)", "rho = nr / np.where(zero, 1.0, nx * nx)"),
    "ratio_zero_token": ("rho[zero] = 0.0", "rho[zero] = 1.0"),
    "gate_tie_fast": ("return ~(rho < eps)", "return rho > eps"),
    "gate_inverted": ("return ~(rho < eps)", "return rho < eps"),
    "fast_wrong_index": ("return G @ M.T", "return (G @ M.T)[:, ::-1]"),
    "slow_wrong_index": ("return X @ W.T", "return X[:, ::-1] @ W.T"),
    "slow_uses_image": ("Y[slow] = slow_path(W, X[slow])", "Y[slow] = fast_path(M, G[slow])"),
    "fast_uses_dense": ("Y[fast] = fast_path(M, G[fast])", "Y[fast] = slow_path(W, X[fast])"),
    "compact_swapped": ("return t[~flags], t[flags]", "return t[flags], t[~flags]"),
    "compact_unstable": ("return t[~flags], t[flags]", "return t[~flags][::-1], t[flags][::-1]"),
    "gram_outer": ("return V.T @ V", "return V.T @ V + 1e-3 * np.eye(V.shape[1])"),
    "spectral_frobenius": ("return float(np.linalg.norm(W, 2))", "return float(np.linalg.norm(W))"),
    "spectral_power_wrong_side": ("v = W.T @ (W @ v)", "v = W @ (W.T @ v)"),
    "spectral_power_few_steps": ("for _ in range(iters):", "for _ in range(3):"),
    "brute_tie": ("slow = not (rho < eps)", "slow = rho > eps"),
    "brute_slow_uses_image": ("Y[t][o] = sum(W[o][i] * x[i] for i in range(d))",
                              "Y[t][o] = sum(M[o][j] * g[j] for j in range(k))"),
    "path_err_sign": ("np.linalg.norm(Yf - Ys, axis=1), np.linalg.norm(Ys, axis=1)",
                      "np.linalg.norm(Yf + Ys, axis=1), np.linalg.norm(Ys, axis=1)"),
    "path_ynorm_of_fast": ("np.linalg.norm(Yf - Ys, axis=1), np.linalg.norm(Ys, axis=1)",
                           "np.linalg.norm(Yf - Ys, axis=1), np.linalg.norm(Yf, axis=1)"),
    "sweep_error_all_tokens": ("e2 = float(np.sum(err[~slow] ** 2))", "e2 = float(np.sum(err ** 2))"),
    "sweep_calls_all_slow": ("calls = [bool(slow[c:c + tokens_per_call].any())",
                             "calls = [bool(slow[c:c + tokens_per_call].all())"),
    "effective_swapped": ("(1.0 - f) * d_out * k + f * d_out * d", "f * d_out * k + (1.0 - f) * d_out * d"),
    "dgks_never_again": ("if np.linalg.norm(v) < eta * before:", "if False:"),
    "dgks_always_again": ("if np.linalg.norm(v) < eta * before:", "if np.linalg.norm(v) <= before:"),
    "dgks_no_normalise": ("Q[:, j] = v / np.linalg.norm(v)", "Q[:, j] = v"),
    "calibration_smallest": ("V = U[:, np.argsort(w)[::-1][:k]]", "V = U[:, np.argsort(w)[:k]]"),
    "calibration_no_sign": ("return V * np.sign(V[piv, np.arange(V.shape[1])])[None, :]", "return V"),
    "subspace_skips_cov": ("return dgks_orthonormalize(X.T @ (X @ V))", "return dgks_orthonormalize(V + 0 * X[:1, :1])"),
    "coherence_not_squared": ("return float(np.sum((Va.T @ Vb) ** 2) / Va.shape[1])",
                              "return float(np.sum(np.abs(Va.T @ Vb)) / Va.shape[1])"),
    "stack_shares_tokens": ("for (W, M, V), X in zip(maps, Xs)]", "for (W, M, V), X in zip(maps, Xs[:1] * len(Xs))]"),
}


def _mutant(old, new):
    assert SRC.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(SRC.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    mod = _mutant(*MUTANTS[name])
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception as e:  # AssertionError or a shape error both count
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"no pin caught mutant {name}"
