"""GPU parity of the tensor-core path below prefill size (T < 128).

There the fast and slow outputs run as few-token contractions on tcgen05:
the weight rows (M or W) are the MMA's 128-row side and the tokens its
narrow side, and the K dimension of the slow one is cut into slices whose
partial tiles are added inside a thread-block cluster.  The finalize (rho,
flags, bf16 g) is split over blocks of Gram rows, and the last CTA to arrive
adds the blocks.  Checked against the float64 oracle on ragged shapes
(d_out not a multiple of 128, K not a multiple of 64) and the decode
shapes, over all-fast, all-slow and mixed calls, with one workspace reused
across token counts.  Definitions: "Gated Subspace Inference for Transformer
Acceleration", §2.1 (decomposition, image) and §2.2 (gate).
"""
import pytest
import torch

from tests.gpu_util import compare
from workloads import synth

pytestmark = pytest.mark.gpu

SHAPES = {"ragged": (1032, 1000, 136), "6b_down": (16384, 4096, 256), "13b_qkv": (5120, 15360, 320)}
CASES = [(1, 1.0), (5, 0.4), (16, 0.25), (17, 0.0), (33, 1.0), (64, 0.3), (127, 0.1)]


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
        V64 = synth.orthonormal_basis(synth.rng(12, d, k, 2), d, k)
        W = synth.storage(synth.gaussian_weight(synth.rng(12, d, k, 1), d_out, d), torch.bfloat16)
        V = synth.storage(V64, torch.bfloat16)
        gm = gsi.make_map(W.cuda(), V.cuda())
        ws = gsi.new_workspace(max(gsi.workspace_size(gm, T, "tensor") for T, _ in CASES))
        _MAPS[name] = (W, V, V64, gm, ws)
    return _MAPS[name]


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("T,f", CASES)
def test_tensor_path_few_tokens(gsi, name, T, f):
    W, V, V64, gm, ws = _map(gsi, name)
    X = synth.map_tokens(12, T, 0, V64, T, f, salt=int(f * 100))
    m_in = synth.MapInputs(f"{name}.T{T}", W, V, X, synth.EPS, V64)
    Y = torch.full((T, gm.d_out), float("nan"), device="cuda")
    Y, flags, rho = gsi.linear(gm, X.cuda(), m_in.eps, Y=Y, workspace=ws, path="tensor")
    st = compare(m_in, gm.M, Y, flags, rho)
    assert gsi.workspace_status(ws) == 0
    n_slow = round(f * T)
    assert abs(st["n_slow"] - n_slow) <= st["n_band"], st
    # every row written (no NaN left from the fill), and run-to-run determinism
    assert not torch.isnan(Y).any()
    Y2, f2, r2 = gsi.linear(gm, X.cuda(), m_in.eps, workspace=ws, path="tensor")
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2) and torch.equal(flags, f2) and torch.equal(rho, r2)


def test_tensor_path_few_tokens_matches_stream_flags(gsi):
    """The same call on the streaming kernels decides the same flags outside
    the tolerance band and gives outputs within the bf16 tolerance."""
    W, V, V64, gm, ws = _map(gsi, "ragged")
    T = 40
    X = synth.map_tokens(12, 77, 0, V64, T, 0.5, salt=7).cuda()
    Yt, ft, rt = gsi.linear(gm, X, synth.EPS, path="tensor")
    Ys, fs, rs = gsi.linear(gm, X, synth.EPS, path="stream")
    torch.cuda.synchronize()
    band = (rs - synth.EPS).abs() <= 1e-3
    assert torch.equal(ft[~band], fs[~band])
    same = (ft == fs)
    rel = (Yt[same] - Ys[same]).norm() / Ys[same].norm()
    assert rel.item() < 2e-2


@pytest.mark.parametrize("T,f", [(3, 1.0), (8, 0.5), (8, 0.0), (200, 0.6)])
def test_stream_path_slow_rows_on_tensor_cores(gsi, T, f):
    """bf16 maps on the two-launch path: the decide-and-apply kernel writes
    the fast rows and the compaction, and the slow rows follow as the
    few-token contraction (T = 200: two tiles of 128 token rows)."""
    W, V, V64, gm, ws = _map(gsi, "ragged")
    X = synth.map_tokens(12, 300 + T, 0, V64, T, f, salt=3)
    m_in = synth.MapInputs(f"ragged.stream.T{T}", W, V, X, synth.EPS, V64)
    wss = gsi.new_workspace(gsi.workspace_size(gm, T, "stream"))
    Y = torch.full((T, gm.d_out), float("nan"), device="cuda")
    Y, flags, rho = gsi.linear(gm, X.cuda(), m_in.eps, Y=Y, workspace=wss, path="stream")
    st = compare(m_in, gm.M, Y, flags, rho)
    assert gsi.workspace_status(wss) == 0
    assert abs(st["n_slow"] - round(f * T)) <= st["n_band"], st
    assert not torch.isnan(Y).any()
