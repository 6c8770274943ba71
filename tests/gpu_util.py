"""Helpers shared by the GPU parity tests: upload seeded inputs, run the
library, and compare with the float64 oracle on the same stored values.

Tolerances (from the arithmetic the kernels do):
  * flags: bit-exact for every token whose oracle rho lies outside
    [eps - 1e-3, eps + 1e-3]; inside that band either decision is correct and
    the output must match the oracle's candidate for the decision taken;
  * rho: |rho_gpu - rho_oracle| <= 2e-4 (float32 accumulation of the exact
    Gram form; the band is 5x wider);
  * Y: relative L2 (||dY||_F / ||Y_ref||_F) <= 1e-5 for float32 maps and
    <= 2e-2 for bf16 maps with float32 accumulation, against the oracle run
    on the same bf16-rounded W, V, X and on the M bytes the library built.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import gsi_oracle as orc
from workloads import synth

BAND = 1e-3
RHO_TOL = 2e-4
TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}


def upload(m_in, dev="cuda"):
    import gated_rank_subspace_gb300 as gsi

    W, V, X = (t.to(dev) for t in (m_in.W, m_in.V, m_in.X))
    return gsi.make_map(W, V), X


def compare(m_in, M_dev, Y, flags, rho, X=None, eps=None, tol=None):
    """Check one call's outputs against the oracle; returns a stats dict."""
    eps = m_in.eps if eps is None else eps
    Wn, Vn = synth.widen(m_in.W), synth.widen(m_in.V)
    Xn = synth.widen(m_in.X if X is None else X)
    Mn = synth.widen(M_dev)
    G = orc.project(Xn, Vn)
    ro = orc.residual_ratio(Xn, orc.residual(Xn, Vn, G))
    fo = orc.gate(ro, eps)
    f = flags.cpu().numpy().astype(bool)
    band = np.abs(ro - eps) <= BAND
    bad = (f != fo) & ~band
    assert not bad.any(), f"flags differ outside the band at tokens {np.nonzero(bad)[0][:10]}"
    if rho is not None:
        r = rho.cpu().numpy().astype(np.float64)
        fin = np.isfinite(ro)
        err = np.max(np.abs(r[fin] - ro[fin])) if fin.any() else 0.0
        assert err <= RHO_TOL, f"rho error {err} > {RHO_TOL}"
        assert np.array_equal(np.isnan(r), np.isnan(ro)), "NaN rho mismatch"
    ref = np.empty((len(f), Wn.shape[0]))
    if (~f).any():
        ref[~f] = orc.fast_path(Mn, G[~f])
    if f.any():
        ref[f] = orc.slow_path(Wn, Xn[f])
    y = Y.cpu().numpy().astype(np.float64)
    fin = np.all(np.isfinite(ref), axis=1)
    num = np.linalg.norm(y[fin] - ref[fin])
    den = np.linalg.norm(ref[fin])
    rel = num / den if den > 0 else num
    tol = TOL[m_in.W.dtype] if tol is None else tol
    assert rel <= tol, f"relative L2 error {rel} > {tol}"
    if (~fin).any():
        assert np.all(np.isnan(y[~fin])), "non-finite tokens must give NaN outputs"
    return dict(rel=rel, n_slow=int(f.sum()), n_band=int(band.sum()), T=len(f))
