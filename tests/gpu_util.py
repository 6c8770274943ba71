"""Helpers shared by the GPU parity tests: upload seeded inputs, run the
library, and compare with the float64 oracle on the same stored values.

Tolerances (from the arithmetic the kernels do):
  * flags: bit-exact for every token whose oracle rho lies outside
    [eps - 1e-3, eps + 1e-3]; inside that band either decision is correct and
    the output must match the oracle's candidate for the decision taken;
  * rho: |rho_gpu^2 - rho_oracle^2| <= 2e-5.  The library forms
    rho^2 = (||x||^2 - 2||g||^2 + g^T Gram g) / ||x||^2 from three float32
    sums of magnitude ~||x||^2 over up to 16384 terms, so the absolute error
    of rho^2 is a few 1e-6 (observed 7.5e-6 at d = 16384); near eps = 0.05
    this bounds |rho error| by 2e-5 / (2 * 0.049) ~= 2e-4, five times inside
    the +-1e-3 band, while at small rho the error in rho itself grows as
    1/rho (harmlessly: such tokens are far from the gate);
  * Y: relative L2 (||dY||_F / ||Y_ref||_F) <= 1e-5 for float32 maps and
    <= 2e-2 for bf16 maps with float32 accumulation, against the oracle run
    on the same bf16-rounded W, V, X and on the M bytes the library built;
    the same bound holds for every token on its own (||dy_t|| / ||y_ref,t||)
    and for every element against its token's RMS output, so a wrong row
    tail or CTA edge cannot hide in the whole-call norm; a token whose
    reference output is exactly zero must come out within that tolerance
    times the median token norm.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import gsi_oracle as orc
from workloads import synth

BAND = 1e-3
RHO2_TOL = 2e-5
TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}


def per_token_rel(y, ref, tol, what="Y"):
    """Per-token checks of an output against its reference; returns the
    largest per-token relative error ||y_t - ref_t|| / ||ref_t||.

    Over the rows with a finite, nonzero reference: that relative error is
    <= tol, and so is every element's error measured against the row's RMS
    (|y_to - ref_to| <= tol * ||ref_t|| / sqrt(d_out)), which catches a few
    wrong or unwritten output rows (a ragged tail, one CTA's rows) that even
    the row norm would average away.  Rows whose reference is exactly zero
    are held to tol * the median row norm."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.all(np.isfinite(ref), axis=1)
    rn = np.linalg.norm(ref, axis=1)
    dn = np.linalg.norm(y - ref, axis=1)
    live = fin & (rn > 0)
    worst = 0.0
    if live.any():
        rel = dn[live] / rn[live]
        worst = float(rel.max())
        bad = np.nonzero(live)[0][rel > tol]
        assert bad.size == 0, f"{what}: per-token relative error {worst} > {tol} at tokens {bad[:10]}"
        rms = rn[live] / np.sqrt(ref.shape[1])
        el = np.max(np.abs(y[live] - ref[live]), axis=1) / rms
        bad = np.nonzero(live)[0][el > tol]
        assert bad.size == 0, (f"{what}: element error {float(el.max())} x the row RMS > {tol} "
                               f"at tokens {bad[:10]}")
    zero = fin & (rn == 0)
    if zero.any():
        scale = float(np.median(rn[fin])) if fin.any() else 0.0
        bad = np.nonzero(zero)[0][dn[zero] > tol * scale]
        assert bad.size == 0, f"{what}: tokens {bad[:10]} should be zero"
    return worst


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
        err = np.max(np.abs(r[fin] ** 2 - ro[fin] ** 2)) if fin.any() else 0.0
        assert err <= RHO2_TOL, f"rho^2 error {err} > {RHO2_TOL}"
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
    worst = per_token_rel(y, ref, tol)
    if (~fin).any():
        # non-finite tokens: the library must reproduce the oracle's pattern
        # (NaN where the exact path gives NaN, the same infinity where it
        # gives +-inf)
        yr, rr = y[~fin], ref[~fin]
        assert np.array_equal(np.isnan(yr), np.isnan(rr)), "NaN pattern of non-finite tokens"
        inf = np.isinf(rr)
        assert np.array_equal(yr[inf], rr[inf]), "infinities of non-finite tokens"
    return dict(rel=rel, worst_token_rel=worst, n_slow=int(f.sum()), n_band=int(band.sum()), T=len(f))
