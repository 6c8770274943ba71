"""The gate's Gram-form residual ratio checked on the device against the
explicit residual x - V_k g ("Gated Subspace Inference for Transformer
Acceleration", §2.1 core decomposition x = V_k g + r; §2.2 rho = ||r|| / ||x||).

gsi_residual_check forms r_t = x_t - V_k g_t with a second pass over V_k from
the projections gsi_gate wrote, and reports each token's explicit ratio and
the largest |rho^2 - rho_explicit^2| over the call.  Checked here: the
explicit ratios against the float64 oracle's (its residual is the definition,
not an identity), the device's maximum against the same figure formed on the
host from the returned arrays, and that maximum within the gate's own
tolerance on rho^2 -- on configs 1 (fp32), 2 (6B maps) and 5 (T = 2048).
"""
import numpy as np
import pytest
import torch

from oracle import gsi_oracle as orc
from tests.gpu_util import RHO2_TOL, upload
from workloads import synth

pytestmark = pytest.mark.gpu

# explicit ratio vs the float64 oracle: float32 dot products of length k and
# sums of squares over d rows, so |rho_x^2 - rho_oracle^2| is a few 1e-7 at most
RHOX2_TOL = 2e-6


@pytest.fixture(scope="module")
def gsi():
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as m

    assert torch.cuda.is_available()
    return m


def _case(name):
    if name == "cfg1":
        return synth.config1()
    if name.startswith("cfg2_"):
        return synth.map_6b(name[5:])
    if name == "cfg5":
        return synth.config5()
    if name == "ragged":
        V64 = synth.orthonormal_basis(synth.rng(8, 1032, 136, 2), 1032, 136)
        return synth.stack_layer(8, 17, {"qkv": V64}, {"qkv": (1000, 1032)}, T=17, f_slow=0.4, roles=("qkv",))[0]
    raise ValueError(name)


@pytest.mark.parametrize("name", ["cfg1", "cfg2_qkv", "cfg2_down", "cfg5", "ragged"])
def test_explicit_residual_matches_gate(gsi, name):
    m_in = _case(name)
    gm, X = upload(m_in)
    G, rho, flags = gsi.gate(gm, X, m_in.eps)
    rho_x, dev = gsi.residual_check(gm, X, G, rho)
    torch.cuda.synchronize()
    Xn, Vn = synth.widen(m_in.X), synth.widen(m_in.V)
    ro = orc.residual_ratio(Xn, orc.residual(Xn, Vn, orc.project(Xn, Vn)))
    rx = rho_x.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(rx ** 2 - ro ** 2)) <= RHOX2_TOL
    r = rho.cpu().numpy().astype(np.float32)
    host = float(np.max(np.abs(r * r - rho_x.cpu().numpy() * rho_x.cpu().numpy())))
    d = float(dev.item())
    assert abs(d - host) <= 1e-9 + 1e-6 * host
    assert d <= RHO2_TOL, f"Gram-form rho^2 deviates from the explicit residual by {d}"
    # bitwise reproducible
    rho_x2, dev2 = gsi.residual_check(gm, X, G, rho)
    torch.cuda.synchronize()
    assert torch.equal(rho_x, rho_x2) and torch.equal(dev, dev2)


def test_zero_and_nonfinite_tokens(gsi):
    V64 = synth.orthonormal_basis(synth.rng(7, 0, 0, 2), 512, 64)
    m_in = synth.stack_layer(7, 0, {"out": V64}, {"out": (384, 512)}, T=6, f_slow=0.5, roles=("out",))[0]
    X = m_in.X.clone()
    X[1] = 0
    X[3, 5] = float("nan")
    gm, _ = upload(m_in)
    Xd = X.cuda()
    G, rho, flags = gsi.gate(gm, Xd, m_in.eps)
    rho_x, dev = gsi.residual_check(gm, Xd, G, rho)
    torch.cuda.synchronize()
    assert float(rho_x[1]) == 0.0
    assert bool(torch.isnan(rho_x[3]))
    assert 0.0 <= float(dev.item()) <= RHO2_TOL
