"""GPU parity of the stack entry point on the 28-layer 6B-shape workload.

28 layers x {QKV, out, MLP up, MLP down} maps with depth-coherent bases
(V^(l+1) = orth(V^(l) + 0.1 N/sqrt(d)), k = 256), bf16 weights, and 512
single-token decode steps whose activations lie near span(V^(l)) with a
per-layer slow fraction f_l ~ U[0.05, 0.15].  Every step runs gsi_stack over
the 112 maps; sampled steps are checked map by map against the float64
oracle.  "Gated Subspace Inference for Transformer Acceleration", §2.2 (the
gate applies to all linear maps) and §2.3 (depth coherence of the bases).
"""
import numpy as np
import pytest
import torch

from tests.gpu_util import compare, per_token_rel
from workloads import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsi():
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as m

    assert torch.cuda.is_available()
    return m


def test_config3_28_layer_stack(gsi):
    L, steps = 28, 512
    bases, fr, base_W, tokens = synth.stack_config3(L, steps)
    dev = "cuda"
    maps, Xs, info = [], [], []
    Wb = {r: base_W[r].to(dev) for r in synth.ROLES}
    for l in range(L):
        for role in synth.ROLES:
            d_out, d = synth.SHAPES_6B[role]
            perm, signs = synth.layer_weight_rows(3, l, synth.ROLE_ID[role], d_out)
            W = (Wb[role][torch.from_numpy(perm).to(dev)] *
                 torch.from_numpy(signs).to(dev, torch.bfloat16)[:, None]).contiguous()
            V = synth.storage(bases[role][l], torch.bfloat16).to(dev)
            maps.append(gsi.make_map(W, V))
            Xs.append(tokens[(l, role)].to(dev))
            info.append((l, role))
    ws = gsi.new_workspace(gsi.stack_workspace_size(maps, 1))
    Ys = [torch.empty(steps, m.d_out, device=dev) for m in maps]
    Fs = [torch.empty(steps, dtype=torch.uint8, device=dev) for _ in maps]
    for t in range(steps):
        args = gsi.stack_args(maps, [X[t:t + 1] for X in Xs], [Y[t:t + 1] for Y in Ys],
                              [F[t:t + 1] for F in Fs])
        gsi.stack_raw(args, len(maps), 1, synth.EPS, ws)
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    # slow fraction per layer follows the recipe (5-15%, sampling noise allowed)
    for l in range(L):
        f = np.mean([Fs[4 * l + j].float().mean().item() for j in range(4)])
        assert 0.02 <= f <= 0.25, (l, f)
    # oracle on sampled steps: gate and fast outputs for every map, the full
    # comparison (slow outputs through the dense W) on three layers
    from oracle import gsi_oracle as orc

    sample = list(range(0, steps, 97)) + [steps - 1]
    idx = torch.tensor(sample)
    for i, (l, role) in enumerate(info):
        X = tokens[(l, role)][sample]
        Y, F = Ys[i][idx].cpu().numpy(), Fs[i][idx].cpu().numpy().astype(bool)
        if l in (0, 13, 27):
            m_in = synth.MapInputs(f"c3.l{l}.{role}", maps[i].W.cpu(), maps[i].V.cpu(), X, synth.EPS)
            compare(m_in, maps[i].M, Ys[i][idx], Fs[i][idx], None)
            continue
        Vn, Xn, Mn = synth.widen(maps[i].V), synth.widen(X), synth.widen(maps[i].M)
        G = orc.project(Xn, Vn)
        ro = orc.residual_ratio(Xn, orc.residual(Xn, Vn, G))
        band = np.abs(ro - synth.EPS) <= 1e-3
        assert np.array_equal(F[~band], orc.gate(ro, synth.EPS)[~band]), (l, role)
        fast = ~F
        if fast.any():
            ref = orc.fast_path(Mn, G[fast])
            rel = np.linalg.norm(Y[fast] - ref) / np.linalg.norm(ref)
            assert rel <= 2e-2, (l, role, rel)
            per_token_rel(Y[fast], ref, 2e-2, f"layer {l} {role}")


@pytest.fixture(scope="module")
def c4(gsi):
    """The 40-layer 13B stack on the device, built once for the module."""
    L = 40
    base_W, V64, rows, cols, pools = synth.stack_config4(L)
    dev = "cuda"
    Wb = {r: base_W[r].to(dev) for r in synth.ROLES}
    Vb = {r: synth.storage(V64[r], torch.bfloat16).to(dev) for r in synth.ROLES}
    maps, info = [], []
    for l in range(L):
        for role in synth.ROLES:
            perm, signs = rows[(l, role)]
            W = (Wb[role][torch.from_numpy(perm).to(dev)] *
                 torch.from_numpy(signs).to(dev, torch.bfloat16)[:, None]).contiguous()
            V = Vb[role][:, torch.from_numpy(cols[(l, role)]).to(dev)].contiguous()
            maps.append(gsi.make_map(W, V))
            info.append((l, role))
    yield maps, info, pools
    del maps
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T,f,steps", [(1, 0.05, 8), (4, 0.05, 4), (16, 0.25, 2)])
def test_config4_40_layer_stack(gsi, c4, T, f, steps):
    """13B shapes, k = 320, 40 layers x 4 maps through gsi_stack, T tokens per
    call with per-token Bernoulli(f) slow labels; every map's gate and the
    first and last layers' outputs against the oracle."""
    L = 40
    maps, info, pools = c4
    n = T * steps
    Xs = [synth.pool_tokens(pools, role, l, n, f, salt=T) for (l, role) in info]
    Xd = [X.cuda() for X in Xs]
    Ys = [torch.empty(n, m.d_out, device="cuda") for m in maps]
    Fs = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in maps]
    ws = gsi.new_workspace(gsi.stack_workspace_size(maps, T))
    for s in range(steps):
        sl = slice(s * T, (s + 1) * T)
        args = gsi.stack_args(maps, [X[sl] for X in Xd], [Y[sl] for Y in Ys], [F[sl] for F in Fs])
        gsi.stack_raw(args, len(maps), T, synth.EPS, ws)
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    from oracle import gsi_oracle as orc

    n_slow = 0
    for i, (l, role) in enumerate(info):
        F = Fs[i].cpu().numpy().astype(bool)
        n_slow += int(F.sum())
        if l in (0, L - 1):
            m_in = synth.MapInputs(f"c4.l{l}.{role}", maps[i].W.cpu(), maps[i].V.cpu(), Xs[i], synth.EPS)
            compare(m_in, maps[i].M, Ys[i], Fs[i], None)
            continue
        Vn, Xn = synth.widen(maps[i].V), synth.widen(Xs[i])
        ro = orc.residual_ratio(Xn, orc.residual(Xn, Vn, orc.project(Xn, Vn)))
        band = np.abs(ro - synth.EPS) <= 1e-3
        assert np.array_equal(F[~band], orc.gate(ro, synth.EPS)[~band]), (l, role)
    # the slow fraction follows the labels (sampling noise allowed)
    frac = n_slow / (n * len(maps))
    assert abs(frac - f) <= 0.05 + 3 * np.sqrt(f * (1 - f) / (n * len(maps))), frac
