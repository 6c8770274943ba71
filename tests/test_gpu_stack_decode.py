"""The persistent stack kernel: gsi_stack_ex(GSI_STACK_PERSISTENT) with one
token per map runs a list of maps in one launch, map after map, with a grid
barrier between them
("Gated Subspace Inference for Transformer Acceleration", §2.2: the gate on
every linear map of a layer -- QKV, output, MLP up and down -- and on every
layer).

Its per-map arithmetic is the single-token kernel's, so its outputs must be
bitwise those of one gsi_linear call per map, and they must match the
float64 oracle within the tolerances of tests/gpu_util.py.  Covered: the
6B layer (cluster projection for qkv, out and up, grid projection for down,
in one launch), fast and slow calls, a list longer than one launch holds,
runs split by element type / width / k, a map the single-token kernel cannot
take in the middle of a list, eps = 0 and eps = inf.
"""
import numpy as np
import pytest
import torch

from tests.gpu_util import compare, upload
from workloads import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsi():
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as m

    assert torch.cuda.is_available()
    return m


def _stack_steps(gsi, maps, Xs, eps, steps):
    """gsi_stack over `maps` once per step, one token per map per step."""
    Ys = [torch.full((steps, m.d_out), float("nan"), device="cuda") for m in maps]
    Fs = [torch.full((steps,), 7, dtype=torch.uint8, device="cuda") for _ in maps]
    ws = gsi.new_workspace(gsi.stack_workspace_size(maps, 1))
    for t in range(steps):
        args = gsi.stack_args(maps, [X[t:t + 1] for X in Xs], [Y[t:t + 1] for Y in Ys], [F[t:t + 1] for F in Fs])
        gsi.stack_raw(args, len(maps), 1, eps, ws, mode="persistent")
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    return Ys, Fs


def _single_calls(gsi, maps, Xs, eps, steps):
    Ys, Fs = [], []
    ws = gsi.new_workspace(max(gsi.workspace_size(m, 1) for m in maps))
    for m, X in zip(maps, Xs):
        Y = torch.empty(steps, m.d_out, device="cuda")
        F = torch.empty(steps, dtype=torch.uint8, device="cuda")
        for t in range(steps):
            gsi.linear(m, X[t:t + 1], eps, Y=Y[t:t + 1], flags=F[t:t + 1], want_rho=False, workspace=ws)
        Ys.append(Y)
        Fs.append(F)
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    return Ys, Fs


def test_6b_layer_in_one_launch_matches_single_calls_and_oracle(gsi):
    steps = 40
    ins = [synth.map_6b(r, T=steps, n_slow=8) for r in synth.ROLES]
    ups = [upload(m) for m in ins]
    maps, Xs = [u[0] for u in ups], [u[1] for u in ups]
    Ys, Fs = _stack_steps(gsi, maps, Xs, synth.EPS, steps)
    Y1, F1 = _single_calls(gsi, maps, Xs, synth.EPS, steps)
    for m_in, gm, Y, F, Ya, Fa in zip(ins, maps, Ys, Fs, Y1, F1):
        assert torch.equal(F, Fa), m_in.name
        assert torch.equal(Y, Ya), m_in.name
        st = compare(m_in, gm.M, Y, F, None)
        assert st["n_slow"] == 8, st
    # bitwise determinism of the persistent launch
    Ys2, _ = _stack_steps(gsi, maps, Xs, synth.EPS, steps)
    for Y, Y2 in zip(Ys, Ys2):
        assert torch.equal(Y, Y2)


@pytest.mark.parametrize("eps", [0.0, float("inf")])
def test_all_slow_and_all_fast(gsi, eps):
    steps = 6
    ins = [synth.map_6b(r, T=steps, n_slow=2) for r in ("out", "down", "qkv")]
    ups = [upload(m) for m in ins]
    maps, Xs = [u[0] for u in ups], [u[1] for u in ups]
    Ys, Fs = _stack_steps(gsi, maps, Xs, eps, steps)
    Y1, F1 = _single_calls(gsi, maps, Xs, eps, steps)
    for m_in, gm, Y, F, Ya, Fa in zip(ins, maps, Ys, Fs, Y1, F1):
        assert bool(F.all()) if eps == 0.0 else not bool(F.any())
        assert torch.equal(Y, Ya) and torch.equal(F, Fa)
        compare(m_in, gm.M, Y, F, None, eps=eps)


def _small_map(seed, d, d_out, k, T, dtype=torch.bfloat16):
    V64 = synth.orthonormal_basis(synth.rng(30, seed, k, 2), d, k)
    m_in = synth.stack_layer(30, seed, {"qkv": V64}, {"qkv": (d_out, d)}, T=T, f_slow=0.3, roles=("qkv",))[0]
    if dtype == torch.float32:
        m_in = synth.MapInputs(m_in.name, m_in.W.float(), m_in.V.float(), m_in.X.float(), m_in.eps, V64)
    return m_in


def test_long_and_mixed_lists(gsi):
    """130 maps: a run of 120 alike (more than one launch holds: 112 + 8),
    then a float32 map, a map with another k, and a map the single-token
    kernel cannot take (a basis too wide for its grid: one call on the other
    kernels), between shorter runs."""
    steps = 3
    ins = []
    for i in range(130):
        if i == 120:
            ins.append(_small_map(i, 512, 200, 32, steps, torch.float32))
        elif i == 123:
            ins.append(_small_map(i, 1024, 96, 64, steps))
        elif i == 126:
            ins.append(_small_map(i, 32768, 64, 64, steps))
        else:
            ins.append(_small_map(i, 512, 136 + 8 * (i % 5), 48, steps))
    ups = [upload(m) for m in ins]
    maps, Xs = [u[0] for u in ups], [u[1] for u in ups]
    Ys, Fs = _stack_steps(gsi, maps, Xs, synth.EPS, steps)
    Y1, F1 = _single_calls(gsi, maps, Xs, synth.EPS, steps)
    for i, (m_in, gm, Y, F, Ya, Fa) in enumerate(zip(ins, maps, Ys, Fs, Y1, F1)):
        assert torch.equal(F, Fa), i
        assert torch.equal(Y, Ya), i
    for i in (0, 111, 112, 119, 120, 121, 123, 126, 129):
        compare(ins[i], maps[i].M, Ys[i], Fs[i], None)
