"""GPU parity: the CUDA library against the float64 oracle on seeded inputs.

Covers every step of the path through the C ABI: image build (M = W V_k and
the Gram), the gate alone, the compaction, the full gated map on the decode
shapes (one token per call, as the benchmark runs them), small-batch mixes of
fast and slow tokens, ragged shapes, the degenerate cases, the stack of maps,
and run-to-run determinism.  Definitions: "Gated Subspace Inference for
Transformer Acceleration", §2.1 (decomposition, image) and §2.2 (gate).
"""
import numpy as np
import pytest
import torch

from oracle import gsi_oracle as orc
from tests.gpu_util import RHO2_TOL, compare, per_token_rel, upload
from workloads import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsi():
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as m

    assert torch.cuda.is_available()
    return m


# ------------------------------------------------------------------ image build
@pytest.mark.parametrize("case", ["cfg1_f32", "6b_out_bf16", "ragged_bf16"])
def test_image_build(gsi, case):
    if case == "cfg1_f32":
        m_in = synth.config1()
    elif case == "6b_out_bf16":
        m_in = synth.map_6b("out", T=1, n_slow=0)
    else:
        m_in = synth.stack_layer(9, 0, {"qkv": synth.orthonormal_basis(synth.rng(9, 0, 0, 2), 200, 24)},
                                 {"qkv": (77, 200)}, T=3, f_slow=0.0, roles=("qkv",))[0]
    gm, _ = upload(m_in)
    torch.cuda.synchronize()
    Wn, Vn = synth.widen(m_in.W), synth.widen(m_in.V)
    Mref = orc.image(Wn, Vn)
    M = synth.widen(gm.M)
    rel = np.linalg.norm(M - Mref) / np.linalg.norm(Mref)
    tol = 1e-6 if m_in.W.dtype == torch.float32 else 4e-3
    assert rel <= tol, rel
    if m_in.W.dtype == torch.bfloat16:
        # RNE of the float32 sum: every element within one bf16 half-ulp (+ fp32 noise)
        half_ulp = np.abs(Mref) * 2.0 ** -8
        assert np.all(np.abs(M - Mref) <= half_ulp + 1e-5)
    G = gm.gram.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(G - orc.gram(Vn))) <= 1e-5


@pytest.mark.parametrize("shape", [(200, 77, 24), (1032, 1000, 136), (5120, 5120, 320), (4096, 16384, 256)])
def test_image_build_tensor_cores(gsi, shape):
    """The tcgen05 image build (bf16) against float64 W V_k and V_k^T V_k, and
    against the CUDA-core build: the same rounding of (differently ordered)
    float32 sums, so the two M differ by at most one bf16 unit in the last
    place (plus float32 noise); the Gram is the CUDA cores' in both (bitwise
    equal)."""
    d, d_out, k = shape
    V64 = synth.orthonormal_basis(synth.rng(11, d, k, 2), d, k)
    m_in = synth.stack_layer(11, d_out, {"qkv": V64}, {"qkv": (d_out, d)}, T=1, f_slow=0.0, roles=("qkv",))[0]
    W, V = m_in.W.cuda(), m_in.V.cuda()
    M_tc, G_tc = gsi.build_image(W, V)
    M_cc, G_cc = gsi.build_image(W, V, tensor_cores=False)
    torch.cuda.synchronize()
    Wn, Vn = synth.widen(m_in.W), synth.widen(m_in.V)
    Mref = orc.image(Wn, Vn)
    M = synth.widen(M_tc)
    assert np.linalg.norm(M - Mref) / np.linalg.norm(Mref) <= 4e-3
    assert np.all(np.abs(M - Mref) <= np.abs(Mref) * 2.0 ** -8 + 1e-5)
    assert np.max(np.abs(G_tc.cpu().numpy().astype(np.float64) - orc.gram(Vn))) <= 1e-5
    # each build is within half a bf16 ulp (+ float32 noise) of the exact
    # image, so the two differ by at most one ulp (+ twice the noise)
    assert np.all(np.abs(M - synth.widen(M_cc)) <= np.abs(Mref) * 2.0 ** -7 + 2e-5)
    assert torch.equal(G_tc, G_cc)
    # the tensor-core build is bitwise reproducible
    M2, G2 = gsi.build_image(W, V)
    torch.cuda.synchronize()
    assert torch.equal(M_tc, M2) and torch.equal(G_tc, G2)


# ------------------------------------------------------------------ gate and compaction
def test_gate_only_config1(gsi):
    m_in = synth.config1()
    gm, X = upload(m_in)
    G, rho, flags = gsi.gate(gm, X, m_in.eps)
    torch.cuda.synchronize()
    Xn, Vn = synth.widen(m_in.X), synth.widen(m_in.V)
    Go = orc.project(Xn, Vn)
    assert np.max(np.abs(G.cpu().numpy() - Go)) <= 1e-5 * np.max(np.abs(Go))
    ro = orc.residual_ratio(Xn, orc.residual(Xn, Vn, Go))
    assert np.max(np.abs(rho.cpu().numpy().astype(np.float64) ** 2 - ro ** 2)) <= RHO2_TOL
    band = np.abs(ro - m_in.eps) <= 1e-3
    f = flags.cpu().numpy().astype(bool)
    assert np.array_equal(f[~band], orc.gate(ro, m_in.eps)[~band])


@pytest.mark.parametrize("T", [0, 1, 31, 32, 33, 100, 2048, 4095, 4096, 4097, 12289])
def test_compact_bit_exact(gsi, T):
    rs = np.random.default_rng(T)
    f = (rs.random(T) < 0.3).astype(np.uint8)
    flags = torch.from_numpy(f).cuda() if T else torch.zeros(0, dtype=torch.uint8, device="cuda")
    idx, counts = gsi.compact(flags)
    torch.cuda.synchronize()
    fast, slow = orc.compact(f.astype(bool))
    c = counts.cpu().numpy()
    assert c[0] == len(fast) and c[1] == len(slow)
    ix = idx.cpu().numpy()
    assert np.array_equal(ix[:len(fast)], fast)
    assert np.array_equal(ix[T:T + len(slow)], slow)


# ------------------------------------------------------------------ full map
def test_config1_fp32(gsi):
    m_in = synth.config1()
    gm, X = upload(m_in)
    Y, flags, rho = gsi.linear(gm, X, m_in.eps)
    st = compare(m_in, gm.M, Y, flags, rho)
    assert 0 < st["n_slow"] < st["T"]
    # the orthonormal identity form (no Gram) is allowed for float32 bases
    gm2 = gsi.Map(gm.W, gm.V, gm.M, None)
    Y2, f2, r2 = gsi.linear(gm2, X, m_in.eps)
    compare(m_in, gm.M, Y2, f2, r2)


@pytest.mark.parametrize("role", synth.ROLES)
def test_config2_decode_single_token_calls(gsi, role):
    """6B map, bf16, 256 sequential T=1 calls through one workspace."""
    m_in = synth.map_6b(role)
    gm, X = upload(m_in)
    T = X.shape[0]
    ws = gsi.new_workspace(gsi.workspace_size(gm, 1))
    Y = torch.empty(T, gm.d_out, device="cuda")
    flags = torch.empty(T, dtype=torch.uint8, device="cuda")
    rho = torch.empty(T, device="cuda")
    for t in range(T):
        gsi.linear(gm, X[t:t + 1], m_in.eps, Y=Y[t:t + 1], flags=flags[t:t + 1], rho=rho[t:t + 1],
                   workspace=ws)
    st = compare(m_in, gm.M, Y, flags, rho)
    assert st["n_slow"] == 26, st
    assert gsi.workspace_status(ws) == 0
    # bitwise determinism: the same call again gives identical bytes
    Y2 = torch.empty_like(Y)
    for t in range(0, T, 37):
        gsi.linear(gm, X[t:t + 1], m_in.eps, Y=Y2[t:t + 1], flags=flags[t:t + 1], workspace=ws)
    torch.cuda.synchronize()
    for t in range(0, T, 37):
        assert torch.equal(Y[t], Y2[t])


@pytest.mark.parametrize("role", synth.ROLES)
def test_config4_small_batch_mix(gsi, role):
    """13B map, k=320, T in {1,4,16} with slow fraction {0, 5, 25, 100}%."""
    d_out, d = synth.SHAPES_13B[role]
    r = synth.ROLE_ID[role]
    V64 = synth.orthonormal_basis(synth.rng(4, 0, r, 2), d, 320)
    W = synth.storage(synth.gaussian_weight(synth.rng(4, 0, r, 1), d_out, d), torch.bfloat16)
    V = synth.storage(V64, torch.bfloat16)
    gm = gsi.make_map(W.cuda(), V.cuda())
    for T in (1, 4, 16):
        for f in (0.0, 0.05, 0.25, 1.0):
            X = synth.map_tokens(4, 0, r, V64, T, f, bernoulli=True, salt=int(T * 1000 + f * 100))
            m_in = synth.MapInputs(f"13b.{role}", W, V, X, synth.EPS, V64)
            Y, flags, rho = gsi.linear(gm, X.cuda(), m_in.eps)
            st = compare(m_in, gm.M, Y, flags, rho)
            if f == 0.0:
                assert st["n_slow"] == 0
            if f == 1.0:
                assert st["n_slow"] == T


@pytest.mark.parametrize("shape", [(200, 77, 24, 5), (200, 77, 24, 33), (64, 300, 8, 9), (1032, 1000, 136, 17)])
def test_ragged_shapes_bf16(gsi, shape):
    d, d_out, k, T = shape
    V64 = synth.orthonormal_basis(synth.rng(8, d, k, 2), d, k)
    m_in = synth.stack_layer(8, T, {"qkv": V64}, {"qkv": (d_out, d)}, T=T, f_slow=0.4, roles=("qkv",))[0]
    gm, X = upload(m_in)
    Y, flags, rho = gsi.linear(gm, X, m_in.eps)
    compare(m_in, gm.M, Y, flags, rho)


# ------------------------------------------------------------------ degenerate cases
def _small_bf16(T=12, f=0.5):
    V64 = synth.orthonormal_basis(synth.rng(7, 0, 0, 2), 512, 64)
    return synth.stack_layer(7, 0, {"out": V64}, {"out": (384, 512)}, T=T, f_slow=f, roles=("out",))[0]


def test_eps_zero_is_dense(gsi):
    m_in = _small_bf16()
    gm, X = upload(m_in)
    Y, flags, rho = gsi.linear(gm, X, 0.0)
    assert bool(flags.all())
    dense = orc.slow_path(synth.widen(m_in.W), synth.widen(m_in.X))
    y = Y.cpu().numpy()
    assert np.linalg.norm(y - dense) / np.linalg.norm(dense) <= 1e-5
    per_token_rel(y, dense, 1e-5)


def test_eps_inf_is_static_projection(gsi):
    m_in = _small_bf16()
    gm, X = upload(m_in)
    Y, flags, rho = gsi.linear(gm, X, float("inf"))
    assert not bool(flags.any())
    compare(m_in, gm.M, Y, flags, rho, eps=float("inf"))


def test_tokens_in_span_are_fast_and_exact(gsi):
    m_in = _small_bf16()
    V64 = m_in.V64
    a = np.random.default_rng(5).standard_normal((9, V64.shape[1]))
    X = synth.storage(a @ V64.T, torch.bfloat16)
    gm, _ = upload(m_in)
    Y, flags, rho = gsi.linear(gm, X.cuda(), 0.05)
    # bf16 rounding of x leaves a residual of ~1e-3 relative: well below eps
    assert not bool(flags.any())
    assert float(rho.max()) < 0.01
    compare(m_in, gm.M, Y, flags, rho, X=X, eps=0.05)


def test_zero_and_nonfinite_tokens(gsi):
    m_in = _small_bf16(T=6)
    X = m_in.X.clone()
    X[1] = 0
    X[3, 5] = float("nan")
    X[4, 0] = float("inf")
    gm, _ = upload(m_in)
    Y, flags, rho = gsi.linear(gm, X.cuda(), m_in.eps)
    torch.cuda.synchronize()
    f = flags.cpu().numpy()
    assert f[1] == 0 and float(rho[1]) == 0.0 and bool((Y[1] == 0).all())
    assert f[3] == 1 and f[4] == 1
    assert bool(torch.isnan(rho[3])) and bool(torch.isnan(Y[3]).all())
    compare(m_in, gm.M, Y, flags, rho, X=X)


def test_scaling_by_power_of_two(gsi):
    m_in = _small_bf16()
    gm, X = upload(m_in)
    Y, flags, rho = gsi.linear(gm, X, m_in.eps)
    Y2, f2, r2 = gsi.linear(gm, X * 4, m_in.eps)
    torch.cuda.synchronize()
    assert torch.equal(flags, f2)
    assert torch.equal(rho, r2)
    assert torch.equal(Y * 4, Y2)


# ------------------------------------------------------------------ stack
def test_stack_matches_single_calls(gsi):
    maps_in = [synth.map_6b(r, T=3, n_slow=1) for r in synth.ROLES]
    ups = [upload(m) for m in maps_in]
    gms = [u[0] for u in ups]
    Xs = [u[1] for u in ups]
    Ys, flags = gsi.stack(gms, Xs, 0.05)
    for m_in, gm, X, Y, f in zip(maps_in, gms, Xs, Ys, flags):
        Y1, f1, r1 = gsi.linear(gm, X, 0.05)
        torch.cuda.synchronize()
        assert torch.equal(Y, Y1) and torch.equal(f, f1)
        compare(m_in, gm.M, Y, f, None)


# ------------------------------------------------------------------ tensor-core path (prefill T)
@pytest.mark.parametrize("shape", [(512, 384, 64, 160, 0.3), (1032, 1000, 136, 300, 0.2), (4096, 4096, 256, 129, 0.1),
                                   (2048, 1000, 320, 160, 0.25), (1024, 512, 512, 136, 0.3),
                                   (1024, 333, 128, 200, 0.3)])
def test_tensor_path_against_oracle_and_stream(gsi, shape):
    """tcgen05 contractions (G = X V, M G_fast, W X_slow) vs the oracle, ragged tiles; k = 320 and
    k = 512 take the finalize's two 256-column passes over the Gram; d_out = 333 (rows that bulk
    copies cannot send) takes the per-tile contraction's store loop for Y_fast, 64 columns at a time."""
    d, d_out, k, T, f = shape
    V64 = synth.orthonormal_basis(synth.rng(10, d, k, 2), d, k)
    m_in = synth.stack_layer(10, T, {"up": V64}, {"up": (d_out, d)}, T=T, f_slow=f, roles=("up",))[0]
    gm, X = upload(m_in)
    Y, flags, rho = gsi.linear(gm, X, m_in.eps, path="tensor")
    st = compare(m_in, gm.M, Y, flags, rho)
    assert 0 < st["n_slow"] < T
    Ys, fs, rs = gsi.linear(gm, X, m_in.eps, path="stream")
    torch.cuda.synchronize()
    same = (flags == fs).float().mean().item()
    assert same > 0.99  # identical outside the tolerance band
    assert gsi.workspace_status(gsi.new_workspace(256)) == 0


def test_config5_prefill_tensor_path(gsi):
    """T=2048, d=4096, d_out=16384, k=256, 410 slow tokens: AUTO takes the tensor cores."""
    m_in = synth.config5()
    gm, X = upload(m_in)
    ws = gsi.new_workspace(gsi.workspace_size(gm, X.shape[0], "auto"))
    Y, flags, rho = gsi.linear(gm, X, m_in.eps, workspace=ws)
    st = compare(m_in, gm.M, Y, flags, rho)
    assert st["n_slow"] == 410, st
    assert gsi.workspace_status(ws) == 0
    # run-to-run determinism of the tensor path
    Y2, f2, r2 = gsi.linear(gm, X, m_in.eps, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2) and torch.equal(flags, f2)


# ------------------------------------------------------------------ single-launch decode (one or two tokens)
@pytest.mark.parametrize("role", ["qkv", "out", "up", "down"])
@pytest.mark.parametrize("T", [1, 2])
def test_fused_decode_against_oracle(gsi, role, T):
    """The single-launch decode: one token per call runs the single-token
    decode kernel (cluster projection for qkv, out and up; grid projection for
    the 16384-wide down map), two tokens the fused decide-and-apply kernel."""
    m_in = synth.map_6b(role, T=24, n_slow=6)
    gm, X = upload(m_in)
    n = X.shape[0]
    ws = gsi.new_workspace(gsi.workspace_size(gm, T, "fused"))
    Y = torch.empty(n, gm.d_out, device="cuda")
    F = torch.empty(n, dtype=torch.uint8, device="cuda")
    R = torch.empty(n, device="cuda")
    Ys = torch.empty_like(Y)
    Fs = torch.empty_like(F)
    for t0 in range(0, n, T):
        sl = slice(t0, t0 + T)
        gsi.linear(gm, X[sl], m_in.eps, Y=Y[sl], flags=F[sl], rho=R[sl], workspace=ws, path="fused")
        gsi.linear(gm, X[sl], m_in.eps, Y=Ys[sl], flags=Fs[sl], want_rho=False, path="stream")
    st = compare(m_in, gm.M, Y, F, R)
    assert st["n_slow"] == 6
    compare(m_in, gm.M, Ys, Fs, None)
    assert gsi.workspace_status(ws) == 0
    # bitwise determinism of the fused kernel
    Y2 = torch.empty_like(Y)
    for t0 in range(0, n, T):
        sl = slice(t0, t0 + T)
        gsi.linear(gm, X[sl], m_in.eps, Y=Y2[sl], flags=F[sl], want_rho=False, workspace=ws, path="fused")
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2)


def test_fused_rejects_what_it_cannot_run(gsi):
    small = synth.map_6b("out", T=4, n_slow=1)
    gm2, X2 = upload(small)
    with pytest.raises(gsi.GsiError):
        gsi.workspace_size(gm2, 4, "fused")  # more than 2 tokens
    d, k = 65536, 512  # one CTA's slab of V (d / 64 rows of 1 KB) does not fit shared memory
    f = lambda *s: torch.zeros(*s, device="cuda", dtype=torch.bfloat16)
    wide = gsi.Map(f(256, d), f(d, k), f(256, k), torch.zeros(k, k, device="cuda"))
    with pytest.raises(gsi.GsiError):
        gsi.workspace_size(wide, 1, "fused")
    assert gsi.workspace_size(wide, 1, "stream") > 0


# ------------------------------------------------------------------ the single-launch decode on edge cases
def _per_call(gsi, gm, X, eps, T_call, path="auto"):
    """Run the map in calls of T_call tokens (one workspace), as a decoder would."""
    n = X.shape[0]
    Y = torch.empty(n, gm.d_out, device="cuda")
    F = torch.empty(n, dtype=torch.uint8, device="cuda")
    R = torch.empty(n, device="cuda")
    ws = gsi.new_workspace(gsi.workspace_size(gm, T_call, path))
    for t0 in range(0, n, T_call):
        sl = slice(t0, min(n, t0 + T_call))
        # each call writes its own buffer: output rows must start 16-byte aligned
        Yc = torch.empty(sl.stop - sl.start, gm.d_out, device="cuda")
        gsi.linear(gm, X[sl], eps, Y=Yc, flags=F[sl], rho=R[sl], workspace=ws, path=path)
        Y[sl] = Yc
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    return Y, F, R


@pytest.mark.parametrize("T_call", [1, 2])
def test_decode_calls_eps_zero_and_inf(gsi, T_call):
    m_in = _small_bf16()
    gm, X = upload(m_in)
    Y, F, R = _per_call(gsi, gm, X, 0.0, T_call)
    assert bool(F.all())
    dense = orc.slow_path(synth.widen(m_in.W), synth.widen(m_in.X))
    assert np.linalg.norm(Y.cpu().numpy() - dense) / np.linalg.norm(dense) <= 1e-5
    per_token_rel(Y.cpu().numpy(), dense, 1e-5)
    Y, F, R = _per_call(gsi, gm, X, float("inf"), T_call)
    assert not bool(F.any())
    Mn = synth.widen(gm.M)
    static = orc.fast_path(Mn, orc.project(synth.widen(m_in.X), synth.widen(m_in.V)))
    assert np.linalg.norm(Y.cpu().numpy() - static) / np.linalg.norm(static) <= 2e-2
    per_token_rel(Y.cpu().numpy(), static, 2e-2)


@pytest.mark.parametrize("T_call", [1, 2])
def test_decode_calls_zero_and_nonfinite_tokens(gsi, T_call):
    m_in = _small_bf16(T=6)
    X = m_in.X.clone()
    X[1] = 0
    X[3, 5] = float("nan")
    X[4, 0] = float("inf")
    gm, _ = upload(m_in)
    Y, F, R = _per_call(gsi, gm, X.cuda(), m_in.eps, T_call)
    f = F.cpu().numpy()
    assert f[1] == 0 and float(R[1]) == 0.0 and bool((Y[1] == 0).all())
    assert f[3] == 1 and f[4] == 1
    assert bool(torch.isnan(R[3])) and bool(torch.isnan(Y[3]).all())
    compare(m_in, gm.M, Y, F, R, X=X)


# (8200, 520, 64): the single-token kernel's grid projection (the basis is too
# wide for one cluster) with a last CTA that holds no V rows and 5 output rows
# per CTA; (16, 8, 8): one V row per rank, partial sums in their own slots
@pytest.mark.parametrize("shape", [(520, 333, 24), (1032, 2056, 40), (16, 8, 8), (8200, 520, 64)])
def test_decode_calls_ragged_shapes(gsi, shape):
    d, d_out, k = shape
    V64 = synth.orthonormal_basis(synth.rng(8, d, k, 3), d, k)
    m_in = synth.stack_layer(8, 1, {"qkv": V64}, {"qkv": (d_out, d)}, T=10, f_slow=0.4, roles=("qkv",))[0]
    gm, X = upload(m_in)
    for T_call in (1, 2):
        Y, F, R = _per_call(gsi, gm, X, m_in.eps, T_call)
        compare(m_in, gm.M, Y, F, R)


def test_decode_calls_fp32(gsi):
    m_in = synth.config1()
    gm, X = upload(m_in)
    Y, F, R = _per_call(gsi, gm, X[:16], m_in.eps, 1)
    compare(m_in, gm.M, Y, F, R, X=m_in.X[:16])
