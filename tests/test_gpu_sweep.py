"""Threshold sweep on the GPU against the float64 oracle.

`gsi_path_errors` gives every token's two candidate outputs (M g and W x),
its residual ratio and the distance between the candidates; `gsi_eps_sweep`
turns those into the gate's slow count, the calls that read W and the
relative output error at each threshold ("Gated Subspace Inference for
Transformer Acceleration", §2.2 and its Theorem 4 bound; §4 static-projection
control).  Tolerances as in tests/gpu_util.py: float32 maps 1e-5, bf16 maps
2e-2 relative; slow counts exact except for tokens whose oracle rho lies within
1e-3 of a threshold.
"""
import numpy as np
import pytest
import torch

from oracle import gsi_oracle as orc
from tests.gpu_util import BAND, RHO2_TOL, TOL, per_token_rel, upload
from workloads import synth

pytestmark = pytest.mark.gpu

EPS_LIST = [0.0, 0.0125, 0.025, 0.05, 0.1, 0.2, 0.4, float("inf")]


@pytest.fixture(scope="module")
def gsi():
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as g

    return g


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def _check_map(gsi, m_in, tokens_per_call=1):
    gm, X = upload(m_in)
    Yf, Ys, rho, err, ynorm = gsi.path_errors(gm, X)
    ns, nc, rel = gsi.eps_sweep(rho, err, ynorm, EPS_LIST, tokens_per_call)
    torch.cuda.synchronize()
    tol = TOL[m_in.W.dtype]
    Wn, Vn, Xn, Mn = (synth.widen(t) for t in (m_in.W, m_in.V, m_in.X, gm.M))
    ro, eo, yo = orc.path_errors(Wn, Mn, Vn, Xn)
    G = orc.project(Xn, Vn)
    # candidates: the fast path for every token, the slow path for every token
    finite = np.isfinite(ro)
    assert _rel(Yf.cpu().numpy()[finite], orc.fast_path(Mn, G)[finite]) <= tol
    assert _rel(Ys.cpu().numpy(), orc.slow_path(Wn, Xn)) <= tol
    per_token_rel(Yf.cpu().numpy()[finite], orc.fast_path(Mn, G)[finite], tol, "Y_fast")
    per_token_rel(Ys.cpu().numpy(), orc.slow_path(Wn, Xn), tol, "Y_slow")
    r = rho.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(r[finite] ** 2 - ro[finite] ** 2)) <= RHO2_TOL
    # per-token distances, relative to the dense output's norm
    e = err.cpu().numpy().astype(np.float64)
    y = ynorm.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(y - yo) / np.maximum(yo, 1e-30)) <= tol
    assert np.max(np.abs(e - eo) / np.maximum(yo, 1e-30)) <= tol
    # the sweep
    want = orc.eps_sweep(ro, eo, yo, EPS_LIST, tokens_per_call)
    ns, nc, rel = ns.cpu().numpy(), nc.cpu().numpy(), rel.cpu().numpy()
    for i, eps in enumerate(EPS_LIST):
        band = int(np.sum(np.abs(ro - eps) <= BAND)) if np.isfinite(eps) else 0
        assert abs(int(ns[i]) - want[i][0]) <= band, f"eps {eps}: slow {ns[i]} vs {want[i][0]}"
        assert abs(int(nc[i]) - want[i][1]) <= band, f"eps {eps}: calls {nc[i]} vs {want[i][1]}"
        if band == 0:
            assert abs(float(rel[i]) - want[i][2]) <= tol * max(want[i][2], 1e-3), f"eps {eps}: error"
    return ro, eo, yo, Wn, Xn, ns, rel


def test_config1_sweep(gsi):
    """fp32 single layer: candidates, ratios, distances and the sweep."""
    ro, eo, yo, Wn, Xn, ns, rel = _check_map(gsi, synth.config1())
    # Theorem 4 on the orthonormal (fp32) basis: ||M g - W x|| <= ||W||_2 rho ||x||
    bound = orc.spectral_norm(Wn) * ro * np.linalg.norm(Xn, axis=1)
    assert np.all(eo <= bound * (1 + 1e-9) + 1e-12)
    assert ns[0] == len(ro) and rel[0] == 0.0, "eps = 0: all slow, exact"
    assert np.all(np.diff(ns.astype(np.int64)) <= 0) and np.all(np.diff(rel) >= 0)


@pytest.mark.parametrize("role", ["out", "down"])
def test_6b_sweep(gsi, role):
    """bf16 6B maps with the two-level token mixture (26 of 64 slow at eps)."""
    _check_map(gsi, synth.map_6b(role, T=64, n_slow=26))


def test_13b_calls_of_16_tokens(gsi):
    """13B-class map (k = 320), Bernoulli(5%) slow labels, calls of 16 tokens:
    a call reads W when any of its tokens is slow."""
    V64 = synth.orthonormal_basis(synth.rng(4, 0, 0, 1), 5120, 320)
    W = synth.gaussian_weight(synth.rng(4, 0, 0, 2), 5120, 5120)
    X = synth.map_tokens(4, 0, 1, V64, 64, 0.05, bernoulli=True)
    m_in = synth.MapInputs("c4.out", synth.storage(W, torch.bfloat16), synth.storage(V64, torch.bfloat16), X,
                           synth.EPS, V64)
    _check_map(gsi, m_in, tokens_per_call=16)


def test_sweep_kernel_by_hand(gsi):
    """The sweep kernel on a hand-worked example: ties slow, NaN slow at every
    threshold, a call (2 tokens) reads W when any of its tokens is slow."""
    dev = "cuda"
    rho = torch.tensor([0.0, 0.3, 0.5, float("nan"), 0.5], device=dev)
    err = torch.tensor([1.0, 2.0, 3.0, 4.0, 5.0], device=dev)
    ynorm = torch.ones(5, device=dev)
    ns, nc, rel = gsi.eps_sweep(rho, err, ynorm, [0.0, 0.3, 0.5, 0.6, float("inf")], tokens_per_call=2)
    assert ns.cpu().tolist() == [5, 4, 3, 1, 1]
    assert nc.cpu().tolist() == [3, 3, 2, 1, 1]
    want = [0.0, np.sqrt(1 / 5), 1.0, np.sqrt(39 / 5), np.sqrt(39 / 5)]
    assert np.allclose(rel.cpu().numpy(), want, rtol=1e-6, atol=0)


def test_sweep_empty_and_reproducible(gsi):
    e = torch.empty(0, device="cuda")
    ns, nc, rel = gsi.eps_sweep(e, e, e, [0.05])
    assert ns.item() == 0 and nc.item() == 0 and rel.item() == 0.0
    m_in = synth.map_6b("out", T=16, n_slow=4)
    gm, X = upload(m_in)
    a = gsi.path_errors(gm, X)
    b = gsi.path_errors(gm, X)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
