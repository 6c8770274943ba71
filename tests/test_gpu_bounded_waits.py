"""Bounded device waits give up, report and recover (no fault, no hang).

The single-token decode kernel's grid projection polls the other clusters'
epoch-tagged slices of g.  The test hook gsi_debug_withhold_slice makes
cluster 0 withhold its slice for one call, so every rank's poll runs out
(after ~10 ms) -- a flag that nothing sets.  The call must still finish, the
workspace's error word must read GSI_ERR_TIMEOUT, and after the workspace is
zeroed again the same call must be correct.  "Gated Subspace Inference for
Transformer Acceleration", §2.2 (the gate this kernel evaluates).
"""
import time

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


def test_withheld_slice_times_out_and_recovers(gsi):
    # d = 8200, k = 64: too wide for one 16-CTA cluster to hold V, so the
    # single-token kernel takes the grid projection
    d, d_out, k = 8200, 520, 64
    V64 = synth.orthonormal_basis(synth.rng(8, d, k, 3), d, k)
    m_in = synth.stack_layer(8, 1, {"qkv": V64}, {"qkv": (d_out, d)}, T=2, f_slow=0.5, roles=("qkv",))[0]
    gm, X = upload(m_in)
    ws = gsi.new_workspace(gsi.workspace_size(gm, 1))
    Y = torch.empty(1, d_out, device="cuda")
    F = torch.empty(1, dtype=torch.uint8, device="cuda")
    R = torch.empty(1, device="cuda")
    gsi.linear(gm, X[:1], m_in.eps, Y=Y, flags=F, rho=R, workspace=ws)
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0

    gsi.lib().gsi_debug_withhold_slice(1)
    t0 = time.perf_counter()
    try:
        gsi.linear(gm, X[:1], m_in.eps, Y=Y, flags=F, rho=R, workspace=ws)
        torch.cuda.synchronize()
    finally:
        gsi.lib().gsi_debug_withhold_slice(0)
    assert time.perf_counter() - t0 < 1.5, "the poll should give up after ~10 ms"
    # the timeout bit (reported as GSI_ERR_TIMEOUT) and the bit naming the
    # wait that gave up: the poll for the other clusters' slices of g
    assert gsi.workspace_status(ws) == 1 | (1 << 11)

    # zero the workspace again; the next calls are correct
    gsi.lib().gsi_workspace_init(ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    Y2 = torch.empty(2, d_out, device="cuda")
    F2 = torch.empty(2, dtype=torch.uint8, device="cuda")
    R2 = torch.empty(2, device="cuda")
    for t in range(2):
        Yc = torch.empty(1, d_out, device="cuda")
        gsi.linear(gm, X[t:t + 1], m_in.eps, Y=Yc, flags=F2[t:t + 1], rho=R2[t:t + 1], workspace=ws)
        Y2[t:t + 1] = Yc
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    compare(m_in, gm.M, Y2, F2, R2)


@pytest.mark.parametrize("shape", [(8200, 520, 64), (16384, 64, 128)])
def test_refused_coresident_grid_falls_back(gsi, shape):
    """Launches refused for co-residency: AUTO still runs every call (on a
    kernel that needs no co-resident grid, at the end the two-launch
    streaming kernels) with the same results.  (8200, 520, 64): the
    single-token kernel's grid projection is refused; (16384, 64, 128): a
    sixteenth of V does not fit one CTA, so both single-launch forms need a
    co-resident grid and an explicit fused call reports the refusal."""
    d, d_out, k = shape
    V64 = synth.orthonormal_basis(synth.rng(8, d, k, 3), d, k)
    m_in = synth.stack_layer(8, 1, {"qkv": V64}, {"qkv": (d_out, d)}, T=4, f_slow=0.5, roles=("qkv",))[0]
    gm, X = upload(m_in)
    ws = gsi.new_workspace(gsi.workspace_size(gm, 1))
    Y = torch.empty(4, d_out, device="cuda")
    F = torch.empty(4, dtype=torch.uint8, device="cuda")
    R = torch.empty(4, device="cuda")
    gsi.lib().gsi_debug_refuse_coresident(1 << 20)
    try:
        for t in range(4):
            Yc = torch.empty(1, d_out, device="cuda")
            gsi.linear(gm, X[t:t + 1], m_in.eps, Y=Yc, flags=F[t:t + 1], rho=R[t:t + 1], workspace=ws)
            Y[t:t + 1] = Yc
        if d == 16384:
            with pytest.raises(gsi.GsiError, match="co-resident"):
                gsi.linear(gm, X[:1], m_in.eps, workspace=ws, path="fused")
    finally:
        gsi.lib().gsi_debug_refuse_coresident(0)
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    compare(m_in, gm.M, Y, F, R)


def test_small_batch_withheld_slice_times_out_and_recovers(gsi):
    """The small-batch kernel (2 <= T <= 16, bf16) exchanges slices of G
    across clusters through the same kind of epoch-tagged words: with cluster
    0 withholding its words the polls give up (~10 ms), the call finishes,
    the workspace reports the timeout and the wait that gave up, and after
    re-initialisation the call is correct.  A refused co-resident launch
    falls back to the earlier kernels with the same results."""
    d, d_out, k = 1032, 1000, 128
    V64 = synth.orthonormal_basis(synth.rng(9, d, k, 3), d, k)
    m_in = synth.stack_layer(9, 1, {"qkv": V64}, {"qkv": (d_out, d)}, T=6, f_slow=0.5, roles=("qkv",))[0]
    gm, X = upload(m_in)
    ws = gsi.new_workspace(gsi.workspace_size(gm, 6, "batch"))
    Y, F, R = gsi.linear(gm, X, m_in.eps, workspace=ws, path="batch")
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0

    gsi.lib().gsi_debug_withhold_slice(1)
    t0 = time.perf_counter()
    try:
        gsi.linear(gm, X, m_in.eps, Y=Y, flags=F, rho=R, workspace=ws, path="batch")
        torch.cuda.synchronize()
    finally:
        gsi.lib().gsi_debug_withhold_slice(0)
    assert time.perf_counter() - t0 < 1.5, "the poll should give up after ~10 ms"
    assert gsi.workspace_status(ws) == 1 | (1 << 11)

    gsi.lib().gsi_workspace_init(ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    Y, F, R = gsi.linear(gm, X, m_in.eps, workspace=ws, path="batch")
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    compare(m_in, gm.M, Y, F, R)

    # a refused co-resident launch: AUTO runs the call on the earlier kernels
    gsi.lib().gsi_debug_refuse_coresident(1 << 20)
    try:
        Y2, F2, R2 = gsi.linear(gm, X, m_in.eps, workspace=ws)
        with pytest.raises(gsi.GsiError, match="co-resident"):
            gsi.linear(gm, X, m_in.eps, workspace=ws, path="batch")
    finally:
        gsi.lib().gsi_debug_refuse_coresident(0)
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    compare(m_in, gm.M, Y2, F2, R2)
