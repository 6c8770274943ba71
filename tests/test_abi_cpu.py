"""The C ABI on a machine without a GPU: the library loads, exports every
declared entry point, sizes workspaces with host arithmetic, and rejects bad
arguments synchronously, before anything touches the device.

Fake device pointers are plain aligned integers: every call here fails
validation (or the injected fault) before any CUDA call could use them.
"""
import ctypes

import pytest

import __graft_entry__

__graft_entry__.build()
import gated_rank_subspace_gb300 as gsi  # noqa: E402

L = gsi.lib()
P = 0x10000  # fake, 256-byte aligned "device" address


def desc(d=4096, d_out=4096, k=256, dtype=gsi.GSI_BF16, W=P, V=P, M=P, gram=P):
    return gsi.MapDesc(d, d_out, k, dtype, W, V, M, gram)


def ws_size(m, T, path=0):
    n = ctypes.c_size_t(0)
    st = L.gsi_linear_workspace_size(ctypes.byref(m), T, path, ctypes.byref(n))
    return st, n.value


def linear(m, T=1, eps=0.05, X=P, Y=P, flags=P, rho=None, ws=P, ws_bytes=1 << 30, path=0):
    return L.gsi_linear_ex(ctypes.byref(m), X, T, eps, Y, flags, rho, ws, ws_bytes, path, None)


def test_exports_every_declared_symbol():
    names = gsi.declared_symbols()
    assert "gsi_linear" in names and "gsi_build_image" in names and "gsi_stack" in names
    for n in names:
        assert hasattr(L, n), f"libgsi.so does not export {n}"


def test_workspace_size_is_host_arithmetic():
    st, n1 = ws_size(desc(), 1)
    assert st == 0 and n1 > 0 and n1 % 256 == 0
    st, n16 = ws_size(desc(), 16)
    assert st == 0 and n16 > n1
    st, nd = ws_size(desc(d=16384), 1)
    assert st == 0 and nd >= n1


@pytest.mark.parametrize("kw,status,needle", [
    (dict(d=0), 1, "positive"),
    (dict(k=8192, d=8192), 2, "GSI_MAX_K"),
    (dict(k=512, d=256), 1, "exceeds d"),
    (dict(k=250), 2, "multiples of 16"),
    (dict(d=4100), 2, "multiples of 16"),
    (dict(dtype=7), 1, "dtype"),
])
def test_bad_shapes(kw, status, needle):
    st = linear(desc(**kw))
    assert st == status
    assert needle in L.gsi_last_error().decode()


def test_bad_pointers_and_eps():
    assert linear(desc(W=0)) == 1 and "map.W is NULL" in L.gsi_last_error().decode()
    assert linear(desc(V=P + 8)) == 1 and "aligned" in L.gsi_last_error().decode()
    assert linear(desc(gram=0)) == 1 and "Gram" in L.gsi_last_error().decode()
    assert linear(desc(), eps=float("nan")) == 1 and "eps" in L.gsi_last_error().decode()
    assert linear(desc(), eps=-0.1) == 1
    assert linear(desc(), X=0) == 1
    assert linear(desc(), Y=P + 4) == 1
    assert linear(desc(), T=-1) == 1
    assert linear(desc(), path=9) == 1


def test_f32_without_gram_is_allowed_to_validate():
    # f32 with gram == NULL means "V is orthonormal": passes validation and
    # then stops at the injected fault (no device call made).
    L.gsi_debug_fail_after(1)
    st = linear(desc(dtype=gsi.GSI_F32, gram=0, d=256, d_out=256, k=16))
    L.gsi_debug_fail_after(0)
    assert st == 3 and "injected" in L.gsi_last_error().decode()


def test_workspace_checks():
    m = desc()
    _, need = ws_size(m, 1)
    assert linear(m, ws=0) == 4
    assert linear(m, ws=P + 16) == 4 and "256-byte" in L.gsi_last_error().decode()
    assert linear(m, ws_bytes=need - 1) == 4 and "needed" in L.gsi_last_error().decode()


def test_zero_tokens_is_a_no_op():
    assert linear(desc(), T=0) == 0
    assert L.gsi_last_error().decode() == ""


def test_injected_fault_reports_cuda_error_without_a_gpu():
    m = desc()
    L.gsi_debug_fail_after(1)
    try:
        st = linear(m)
    finally:
        L.gsi_debug_fail_after(0)
    assert st == 3
    assert "injected" in L.gsi_last_error().decode()


def test_stack_validation_names_the_map():
    maps = (gsi.MapDesc * 2)(desc(), desc(k=250))
    vp = ctypes.c_void_p
    X = (vp * 2)(P, P)
    Y = (vp * 2)(P, P)
    F = (vp * 2)(P, P)
    st = L.gsi_stack(maps, 2, X, 1, 0.05, Y, F, P, 1 << 30, None)
    assert st == 2 and "map 1" in L.gsi_last_error().decode()
    n = ctypes.c_size_t(0)
    maps_ok = (gsi.MapDesc * 2)(desc(), desc(d=16384))
    assert L.gsi_stack_workspace_size(maps_ok, 2, 1, ctypes.byref(n)) == 0
    _, n2 = ws_size(desc(d=16384), 1)
    assert n.value == n2


def test_build_image_validation():
    st = L.gsi_build_image(P, P, 0, None, 4096, 4096, 256, gsi.GSI_BF16, None)
    assert st == 1 and "M is NULL" in L.gsi_last_error().decode()
    st = L.gsi_build_image(P, P, P, None, 4096, 4096, 250, gsi.GSI_BF16, None)
    assert st == 2


def test_compact_validation():
    assert L.gsi_compact(0, 4, P, P, None) == 1
    assert L.gsi_compact(P, -1, P, P, None) == 1


def test_path_errors_validation():
    m = desc()
    _, need = ws_size(m, 4)

    def call(T=4, rho=P, err=P, ynorm=P, flags=P, ws_bytes=need):
        return L.gsi_path_errors(ctypes.byref(m), P, T, P, P, flags, rho, err, ynorm, P, ws_bytes, None)

    assert call(T=0) == 0
    assert call(rho=None) == 1 and "aligned" in L.gsi_last_error().decode()
    assert call(ynorm=P + 2) == 1
    assert call(flags=None) == 1
    assert call(ws_bytes=need - 1) == 4
    L.gsi_debug_fail_after(1)
    try:
        assert call() == 3 and "injected" in L.gsi_last_error().decode()
    finally:
        L.gsi_debug_fail_after(0)


def test_eps_sweep_validation():
    def call(T=8, n_eps=3, tpc=1, eps=P, out=P, rho=P):
        return L.gsi_eps_sweep(rho, P, P, T, eps, n_eps, tpc, out, P, P, None)

    assert call(n_eps=0) == 0
    assert call(tpc=0) == 1 and "tokens_per_call" in L.gsi_last_error().decode()
    assert call(T=-1) == 1
    assert call(n_eps=70000) == 2
    assert call(eps=None) == 1
    assert call(out=None) == 1
    assert call(rho=None) == 1
