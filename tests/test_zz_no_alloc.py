"""gsi_linear_noalloc: the gated map for callers that cannot allocate.

Callers such as allocator hooks or plug-ins inside a host program that owns
all device memory cannot hand the library a workspace.  The allocation-free
entry point keeps its scratch in a built-in device array instead; these
tests call it through the C ABI and check it against gsi_linear (the entry
point that takes a caller workspace), on two calls in a row that leave
different contents in the shared array, within the tolerances the other
GPU tests use.  The file is named to be collected last.
"""
import ctypes

import pytest
import torch

from tests.gpu_util import compare, per_token_rel, upload
from workloads import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsi():
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as m

    assert torch.cuda.is_available()
    L = m.lib()
    vp = ctypes.c_void_p
    L.gsi_linear_noalloc.argtypes = [ctypes.POINTER(m.MapDesc), vp, ctypes.c_int64, ctypes.c_float,
                                     vp, vp, vp, vp]
    L.gsi_linear_noalloc.restype = ctypes.c_int
    L.gsi_linear_noalloc_max_bytes.argtypes = []
    L.gsi_linear_noalloc_max_bytes.restype = ctypes.c_size_t
    return m


def _noalloc(gsi, gm, X, eps):
    T = X.shape[0]
    Y = torch.full((T, gm.d_out), float("nan"), device="cuda")
    flags = torch.full((T,), 7, dtype=torch.uint8, device="cuda")
    rho = torch.full((T,), -1.0, device="cuda")
    desc = gm.desc()
    st = gsi.lib().gsi_linear_noalloc(ctypes.byref(desc), X.data_ptr(), T, eps, Y.data_ptr(),
                                      flags.data_ptr(), rho.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
    assert st == 0, gsi.lib().gsi_last_error().decode()
    return Y, flags, rho


def test_noalloc_matches_workspace_entry_point_on_two_calls(gsi):
    # call 1: a 6B MLP-down map (d = 16384), 3 tokens; call 2: a 6B QKV map,
    # 5 tokens.  The second call runs on the scratch the first one left.
    cases = [synth.map_6b("down", T=3, n_slow=1), synth.map_6b("qkv", T=5, n_slow=2)]
    for m_in in cases:
        gm, X = upload(m_in)
        Yn, fn, rn = _noalloc(gsi, gm, X, m_in.eps)
        Yw, fw, rw = gsi.linear(gm, X, m_in.eps, path="stream")
        torch.cuda.synchronize()
        assert torch.equal(fn, fw)
        rel = (torch.linalg.norm(Yn - Yw) / torch.linalg.norm(Yw)).item()
        assert rel <= 2e-2, rel
        per_token_rel(Yn.cpu().numpy(), Yw.cpu().numpy(), 2e-2, "noalloc vs workspace")
        assert torch.allclose(rn, rw, rtol=0, atol=1e-6)
        compare(m_in, gm.M, Yn, fn, rn)
        # the built-in scratch's error word: no bounded wait gave up
        code = ctypes.c_uint32(7)
        st = gsi.lib().gsi_linear_noalloc_status(ctypes.byref(code), torch.cuda.current_stream().cuda_stream)
        assert st == 0 and code.value == 0, gsi.lib().gsi_last_error().decode()


def test_noalloc_rejects_calls_beyond_its_scratch(gsi):
    m_in = synth.map_6b("out", T=1, n_slow=0)
    gm, _ = upload(m_in)
    limit = gsi.lib().gsi_linear_noalloc_max_bytes()
    T = 1
    while gsi.workspace_size(gm, T, "stream") <= limit:
        T *= 2
    X = torch.zeros(T, gm.d, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(T, gm.d_out, device="cuda")
    flags = torch.empty(T, dtype=torch.uint8, device="cuda")
    desc = gm.desc()
    st = gsi.lib().gsi_linear_noalloc(ctypes.byref(desc), X.data_ptr(), T, 0.05, Y.data_ptr(),
                                      flags.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert st == 4
    assert "built-in area" in gsi.lib().gsi_last_error().decode()
