"""Basis construction on the GPU against the float64 oracle.

"Gated Subspace Inference for Transformer Acceleration", §2.3 depth cascade
and calibration (readings in the oracle and in include/gsi.h): DGKS
Gram-Schmidt, the correction step V <- DGKS(X^T X V), subspace coherence and
the export to a map's bf16 layout.  The library computes in float32 (the
calibration block may be bf16); tolerances follow from that: orthonormal
vectors agree with the float64 oracle to ~1e-5 relative, coherences to 1e-5.
"""
import numpy as np
import pytest
import torch

from oracle import gsi_oracle as orc
from workloads import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsi():
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as g

    return g


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_dgks_matches_oracle(gsi):
    A = synth.random_basis_t(9, 24, 1000)  # k x d rows
    Vt, n = gsi.basis_orthonormalize(torch.tensor(A, dtype=torch.float32, device="cuda"))
    Q, n_o = orc.dgks_orthonormalize(A.astype(np.float32).astype(np.float64).T)
    got = Vt.cpu().numpy().astype(np.float64)
    assert _rel(got, Q.T) <= 2e-5
    assert int(n.item()) == n_o == 0
    assert np.abs(got @ got.T - np.eye(24)).max() <= 2e-6


def test_dgks_reorthogonalises_near_dependent_rows(gsi):
    A = synth.random_basis_t(9, 16, 2048, salt=1)
    A[5] = A[4] + 1e-4 * A[5]  # row 5 is almost row 4: one projection leaves ~1e-4 of it
    A = A.astype(np.float32).astype(np.float64)
    Vt, n = gsi.basis_orthonormalize(torch.tensor(A, dtype=torch.float32, device="cuda"))
    Q, n_o = orc.dgks_orthonormalize(A.T)
    got = Vt.cpu().numpy().astype(np.float64)
    assert int(n.item()) == n_o == 1
    assert np.abs(got @ got.T - np.eye(16)).max() <= 5e-6
    # the nearly dependent row is determined only to float32 precision / 1e-4
    keep = [i for i in range(16) if i != 5]
    assert _rel(got[keep], Q.T[keep]) <= 5e-5


@pytest.mark.parametrize("xdt", [torch.float32, torch.bfloat16])
def test_step_matches_oracle(gsi, xdt):
    U, blocks = synth.calibration_stream(9, 1, d=384, m=48, T=256)
    X = synth.storage(blocks[0], xdt)
    Xn = synth.widen(X)
    k = 16
    V0 = orc.dgks_orthonormalize(synth.random_basis_t(9, k, 384, salt=2).T)[0]  # d x k
    Vt = torch.tensor(V0.T.copy(), dtype=torch.float32, device="cuda")
    Vt, n = gsi.basis_step(X.cuda(), Vt)
    V1, n_o = orc.subspace_step(Xn, V0.astype(np.float32).astype(np.float64))
    got = Vt.cpu().numpy().astype(np.float64)
    assert _rel(got, V1.T) <= 1e-4
    assert int(n.item()) == n_o


def test_steps_reach_the_principal_subspace(gsi):
    """Repeated steps converge to the oracle's calibration basis; started from
    the previous layer's basis (the cascade) they need fewer steps than from
    a random start."""
    d, m, k, T = 512, 64, 16, 1024
    U, blocks = synth.calibration_stream(9, 2, d=d, m=m, T=T, decay=0.9)
    Xs = [synth.storage(b, torch.float32) for b in blocks]
    refs = [orc.calibration_basis(synth.widen(X), k) for X in Xs]

    def steps_to(X, Vt, ref, target=0.999, cap=60):
        Xd = X.cuda()
        for it in range(1, cap + 1):
            gsi.basis_step(Xd, Vt)
            c = gsi.basis_coherence(Vt, torch.tensor(ref.T.copy(), dtype=torch.float32, device="cuda")).item()
            if c >= target:
                return it, Vt
        return cap + 1, Vt

    Vt0 = torch.tensor(synth.random_basis_t(9, k, d, salt=3), dtype=torch.float32, device="cuda")
    gsi.basis_orthonormalize(Vt0)
    n0, V_l0 = steps_to(Xs[0], Vt0, refs[0])
    assert n0 <= 60, "layer 0 did not converge"
    Vt1 = torch.tensor(synth.random_basis_t(9, k, d, salt=4), dtype=torch.float32, device="cuda")
    gsi.basis_orthonormalize(Vt1)
    n_cold, _ = steps_to(Xs[1], Vt1, refs[1])
    n_warm, _ = steps_to(Xs[1], V_l0.clone(), refs[1])
    assert n_warm < n_cold, f"warm start {n_warm} steps, cold {n_cold}"


def test_coherence_and_export(gsi):
    a = orc.dgks_orthonormalize(synth.random_basis_t(9, 12, 300, salt=5).T)[0]
    b = orc.dgks_orthonormalize(a + 0.3 * synth.random_basis_t(9, 12, 300, salt=6).T)[0]
    ta = torch.tensor(a.T.copy(), dtype=torch.float32, device="cuda")
    tb = torch.tensor(b.T.copy(), dtype=torch.float32, device="cuda")
    c = gsi.basis_coherence(ta, tb).item()
    want = orc.coherence(a.astype(np.float32).astype(np.float64), b.astype(np.float32).astype(np.float64))
    assert abs(c - want) <= 1e-5
    assert abs(gsi.basis_coherence(ta, ta).item() - 1.0) <= 1e-5
    V = gsi.basis_export(ta, torch.bfloat16)
    assert torch.equal(V.cpu(), ta.t().contiguous().cpu().to(torch.bfloat16))
    V32 = gsi.basis_export(ta, torch.float32)
    assert torch.equal(V32, ta.t().contiguous())
