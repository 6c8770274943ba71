"""GPU parity of the small-batch decode kernel (bf16 maps, 2 <= T <= 16).

One launch per call: every CTA projects its slab of V_k on all T tokens, the
clusters exchange slices of G through epoch-tagged words in the workspace,
every CTA takes the same flags from the Gram form of the residual, and the
three products (X V_k, G M^T, X W^T) run as warp-level tensor-core products
with float32 accumulation.  Checked against the float64 oracle on the 6B and
13B map shapes and on ragged ones (d_out not a multiple of 16 rows a CTA, d
not a multiple of the 128-column ring stage, a map smaller than one tile a
CTA), over all-fast, all-slow and mixed calls, with per-token and
per-element bounds, run-to-run determinism, and one workspace shared with the
single-token decode kernel (whose epoch-tagged words sit in the same
workspace).  Definitions: "Gated
Subspace Inference for Transformer Acceleration", §2.1 (decomposition,
image) and §2.2 (gate).
"""
import numpy as np
import pytest
import torch

from oracle import gsi_oracle as orc
from tests.gpu_util import compare
from workloads import synth

pytestmark = pytest.mark.gpu

SHAPES = {
    "ragged": (1032, 1000, 128),     # d % 128 != 0, d_out / 112 CTAs not a multiple of 16
    "small": (128, 40, 64),          # fewer rows than one tile a CTA, a single ring stage
    "6b_up": (4096, 16384, 256),     # 160 output rows a CTA (the most row tiles)
    "6b_down": (16384, 4096, 256),   # the widest slab of V_k
    "13b_qkv": (5120, 15360, 320),   # k = 320: five 64-column boxes
}
CASES = [(2, 0.5), (3, 1.0), (4, 0.25), (8, 0.0), (9, 0.5), (16, 0.25), (16, 1.0)]


@pytest.fixture(scope="module")
def gsi():
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as m

    assert torch.cuda.is_available()
    return m


_MAPS = {}


def _map(gsi, name):
    if name not in _MAPS:
        _MAPS.clear()  # one shape's weights on the device at a time
        d, d_out, k = SHAPES[name]
        V64 = synth.orthonormal_basis(synth.rng(14, d, k, 2), d, k)
        W = synth.storage(synth.gaussian_weight(synth.rng(14, d, k, 1), d_out, d), torch.bfloat16)
        V = synth.storage(V64, torch.bfloat16)
        gm = gsi.make_map(W.cuda(), V.cuda())
        ws = gsi.new_workspace(max(max(gsi.workspace_size(gm, T, "batch") for T, _ in CASES),
                                   gsi.workspace_size(gm, 1)))
        _MAPS[name] = (W, V, V64, gm, ws)
    return _MAPS[name]


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("T,f", CASES)
def test_batch_decode(gsi, name, T, f):
    W, V, V64, gm, ws = _map(gsi, name)
    X = synth.map_tokens(14, T, 0, V64, T, f, salt=int(f * 100))
    m_in = synth.MapInputs(f"{name}.T{T}", W, V, X, synth.EPS, V64)
    Y = torch.full((T, gm.d_out), float("nan"), device="cuda")
    Y, flags, rho = gsi.linear(gm, X.cuda(), m_in.eps, Y=Y, workspace=ws, path="batch")
    st = compare(m_in, gm.M, Y, flags, rho)
    assert gsi.workspace_status(ws) == 0
    assert abs(st["n_slow"] - round(f * T)) <= st["n_band"], st
    # every row written (no NaN left from the fill), and run-to-run determinism
    assert not torch.isnan(Y).any()
    Y2, f2, r2 = gsi.linear(gm, X.cuda(), m_in.eps, workspace=ws, path="batch")
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2) and torch.equal(flags, f2) and torch.equal(rho, r2)


@pytest.mark.parametrize("name", ["ragged", "13b_qkv"])
def test_batch_decode_eps_zero_and_inf(gsi, name):
    """eps = 0: every token exact (Y = X W^T); eps = inf: every token on the
    image (static projection)."""
    W, V, V64, gm, ws = _map(gsi, name)
    T = 11
    X = synth.map_tokens(14, 500, 0, V64, T, 0.5, salt=9)
    Wn, Xn = synth.widen(W), synth.widen(X)
    Y, flags, _ = gsi.linear(gm, X.cuda(), 0.0, workspace=ws, path="batch")
    assert int(flags.sum()) == T
    ref = orc.slow_path(Wn, Xn)
    y = Y.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(y - ref) / np.linalg.norm(ref) <= 2e-2
    m_in = synth.MapInputs(f"{name}.inf", W, V, X, float("inf"), V64)
    Y, flags, rho = gsi.linear(gm, X.cuda(), float("inf"), workspace=ws, path="batch")
    assert int(flags.sum()) == 0
    compare(m_in, gm.M, Y, flags, rho, eps=float("inf"))
    assert gsi.workspace_status(ws) == 0


def test_batch_decode_zero_and_nonfinite_tokens(gsi):
    """A zero token is fast with y = 0 (rho := 0); a token holding inf or NaN
    takes the exact path (rho = NaN) and its NaN reaches only its own row."""
    W, V, V64, gm, ws = _map(gsi, "ragged")
    T = 6
    X = synth.map_tokens(14, 600, 0, V64, T, 0.0, salt=5).clone()
    X[1] = 0
    X[3, 7] = float("nan")
    X[4, 100] = float("inf")
    m_in = synth.MapInputs("ragged.nonfinite", W, V, X, synth.EPS, V64)
    Y, flags, rho = gsi.linear(gm, X.cuda(), synth.EPS, workspace=ws, path="batch")
    compare(m_in, gm.M, Y, flags, rho)
    f = flags.cpu().numpy()
    assert f[1] == 0 and f[3] == 1 and f[4] == 1
    y = Y.cpu().numpy()
    assert np.all(y[1] == 0)
    for t in (0, 2, 5):
        assert np.all(np.isfinite(y[t]))


def test_batch_decode_shares_workspace_with_single_token_calls(gsi):
    """The single-token decode kernel (grid projection on this map) and the
    small-batch kernel alternate on one workspace: each kernel's epoch-tagged
    words carry its own tag, so neither accepts the other's stale words."""
    W, V, V64, gm, ws = _map(gsi, "6b_down")
    X = synth.map_tokens(14, 700, 0, V64, 12, 0.25, salt=2)
    m_in = synth.MapInputs("6b_down.alt", W, V, X, synth.EPS, V64)
    Xd = X.cuda()
    Y = torch.full((12, gm.d_out), float("nan"), device="cuda")
    flags = torch.empty(12, dtype=torch.uint8, device="cuda")
    rho = torch.empty(12, device="cuda")
    for rep in range(3):
        gsi.linear(gm, Xd[0:4], synth.EPS, Y=Y[0:4], flags=flags[0:4], rho=rho[0:4], workspace=ws, path="batch")
        for t in range(4, 8):
            gsi.linear(gm, Xd[t:t + 1], synth.EPS, Y=Y[t:t + 1], flags=flags[t:t + 1], rho=rho[t:t + 1],
                       workspace=ws)
        gsi.linear(gm, Xd[8:12], synth.EPS, Y=Y[8:12], flags=flags[8:12], rho=rho[8:12], workspace=ws, path="batch")
    assert gsi.workspace_status(ws) == 0
    compare(m_in, gm.M, Y, flags, rho)


def test_batch_auto_path_and_stack(gsi):
    """AUTO takes the small-batch kernel for bf16 maps at 2 <= T <= 16; a
    stack of maps of different shapes (one launch each, chained) matches one
    call per map bitwise."""
    maps, Xs = [], []
    for role, (d, d_out) in (("a", (1032, 1000)), ("b", (512, 2056)), ("c", (2048, 520))):
        V64 = synth.orthonormal_basis(synth.rng(15, d, 64, 2), d, 64)
        W = synth.storage(synth.gaussian_weight(synth.rng(15, d, 64, 1), d_out, d), torch.bfloat16)
        maps.append(gsi.make_map(W.cuda(), synth.storage(V64, torch.bfloat16).cuda()))
        Xs.append(synth.map_tokens(15, d, 1, V64, 5, 0.4, salt=1).cuda())
    ws = gsi.new_workspace(gsi.stack_workspace_size(maps, 5))
    Ys = [torch.zeros(5, m.d_out, device="cuda") for m in maps]
    Fs = [torch.zeros(5, dtype=torch.uint8, device="cuda") for _ in maps]
    gsi.stack(maps, Xs, synth.EPS, Ys=Ys, flags=Fs, workspace=ws)
    for m, X, Ysk, Fsk in zip(maps, Xs, Ys, Fs):
        Y1, F1, _ = gsi.linear(m, X, synth.EPS, workspace=ws, path="batch")
        torch.cuda.synchronize()
        assert torch.equal(Y1, Ysk) and torch.equal(F1, Fsk)
    assert gsi.workspace_status(ws) == 0
