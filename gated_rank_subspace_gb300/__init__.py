"""Python binding of libgsi, the gated-subspace linear map on one sm_103a GPU.

The method ("Gated Subspace Inference for Transformer Acceleration",
gist.science technical summary, §2.1-§2.2): for a map W and an orthonormal
basis V_k, each token x is projected, g = V_k^T x; its residual ratio
rho = ||x - V_k g|| / ||x|| decides the path: rho < eps gives the fast path
y = M g with the cached image M = W V_k, otherwise the exact y = W x.

This module only marshals arguments: every step runs in the library's CUDA
kernels (include/gsi.h documents the C ABI).  PyTorch supplies device memory
and streams.  There is no CPU fallback: if libgsi.so has not been built, or
no GPU is present, calls fail loudly.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgsi.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "gsi.h")

GSI_F32, GSI_BF16 = 0, 1
PATHS = {"auto": 0, "stream": 1, "tensor": 2, "fused": 3, "batch": 4}
STATUS = {0: "GSI_OK", 1: "GSI_ERR_INVALID_ARG", 2: "GSI_ERR_UNSUPPORTED", 3: "GSI_ERR_CUDA",
          4: "GSI_ERR_WORKSPACE", 5: "GSI_ERR_TIMEOUT"}


class GsiError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


class MapDesc(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int64), ("d_out", ctypes.c_int64), ("k", ctypes.c_int64),
                ("dtype", ctypes.c_int), ("W", ctypes.c_void_p), ("V", ctypes.c_void_p),
                ("M", ctypes.c_void_p), ("gram", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libgsi.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(or python -m gated_rank_subspace_gb300._build)")
    L = ctypes.CDLL(LIB_PATH)
    i64, vp, f32, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "gsi_build_image": [vp, vp, vp, vp, i64, i64, i64, ctypes.c_int, vp],
        "gsi_build_image_ex": [vp, vp, vp, vp, i64, i64, i64, ctypes.c_int, vp, sz, vp],
        "gsi_linear_workspace_size": [P(MapDesc), i64, ctypes.c_int, P(sz)],
        "gsi_workspace_init": [vp, sz, vp],
        "gsi_workspace_status": [vp, P(ctypes.c_uint32), vp],
        "gsi_gate": [P(MapDesc), vp, i64, f32, vp, vp, vp, vp, sz, vp],
        "gsi_compact": [vp, i64, vp, vp, vp],
        "gsi_apply": [P(MapDesc), vp, vp, i64, vp, vp, sz, vp],
        "gsi_linear": [P(MapDesc), vp, i64, f32, vp, vp, vp, vp, sz, vp],
        "gsi_linear_ex": [P(MapDesc), vp, i64, f32, vp, vp, vp, vp, sz, ctypes.c_int, vp],
        "gsi_stack_workspace_size": [P(MapDesc), i64, i64, P(sz)],
        "gsi_stack": [P(MapDesc), i64, P(vp), i64, f32, P(vp), P(vp), vp, sz, vp],
        "gsi_stack_ex": [P(MapDesc), i64, P(vp), i64, f32, P(vp), P(vp), vp, sz, ctypes.c_int, vp],
        "gsi_path_errors": [P(MapDesc), vp, i64, vp, vp, vp, vp, vp, vp, vp, sz, vp],
        "gsi_eps_sweep": [vp, vp, vp, i64, vp, i64, i64, vp, vp, vp, vp],
        "gsi_basis_orthonormalize": [vp, i64, i64, vp, vp],
        "gsi_basis_step": [vp, ctypes.c_int, i64, i64, i64, vp, vp, sz, vp, vp],
        "gsi_basis_coherence": [vp, vp, i64, i64, vp, vp, vp],
        "gsi_basis_export": [vp, i64, i64, vp, ctypes.c_int, vp],
        "gsi_residual_check": [P(MapDesc), vp, i64, vp, vp, vp, vp, vp, sz, vp],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.gsi_build_image_work_bytes.argtypes = [i64, i64, ctypes.c_int]
    L.gsi_build_image_work_bytes.restype = sz
    L.gsi_residual_check_work_bytes.argtypes = [i64, i64]
    L.gsi_residual_check_work_bytes.restype = sz
    L.gsi_basis_step_work_bytes.argtypes = [i64, i64, i64]
    L.gsi_basis_step_work_bytes.restype = sz
    L.gsi_last_error.argtypes = []
    L.gsi_last_error.restype = ctypes.c_char_p
    L.gsi_debug_fail_after.argtypes = [ctypes.c_int]
    L.gsi_debug_fail_after.restype = None
    L.gsi_debug_withhold_slice.argtypes = [ctypes.c_int]
    L.gsi_debug_withhold_slice.restype = None
    L.gsi_debug_refuse_coresident.argtypes = [ctypes.c_int]
    L.gsi_debug_refuse_coresident.restype = None
    L.gsi_linear_noalloc.argtypes = [P(MapDesc), vp, i64, f32, vp, vp, vp, vp]
    L.gsi_linear_noalloc.restype = ctypes.c_int
    L.gsi_linear_noalloc_max_bytes.argtypes = []
    L.gsi_linear_noalloc_max_bytes.restype = sz
    L.gsi_linear_noalloc_status.argtypes = [P(ctypes.c_uint32), vp]
    L.gsi_linear_noalloc_status.restype = ctypes.c_int
    _lib = L
    return L


def declared_symbols() -> list:
    """Entry points declared in include/gsi.h."""
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(gsi_\w+)\s*\(", src, re.M)))


def _check(status: int):
    if status != 0:
        raise GsiError(status, lib().gsi_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return GSI_F32
    if dt == torch.bfloat16:
        return GSI_BF16
    raise TypeError(f"unsupported dtype {dt}: float32 or bfloat16")


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


@dataclass
class Map:
    """One linear map with its cached artefacts (device tensors).

    W: d_out x d, V: d x k, M: d_out x k (same dtype), gram: k x k float32.
    """
    W: torch.Tensor
    V: torch.Tensor
    M: torch.Tensor
    gram: torch.Tensor

    @property
    def d(self):
        return self.W.shape[1]

    @property
    def d_out(self):
        return self.W.shape[0]

    @property
    def k(self):
        return self.V.shape[1]

    def desc(self) -> MapDesc:
        return MapDesc(self.d, self.d_out, self.k, _dtype_code(self.W.dtype), self.W.data_ptr(),
                       self.V.data_ptr(), self.M.data_ptr(),
                       self.gram.data_ptr() if self.gram is not None else None)


def build_image(W: torch.Tensor, V: torch.Tensor, M=None, gram=None, with_gram=True, stream=None,
                tensor_cores=True):
    """M = W V (and the Gram V^T V) on the GPU; returns (M, gram).  bf16 maps
    use the tensor cores (a scratch area is allocated here, by PyTorch)
    unless tensor_cores is False, which keeps the CUDA-core kernel."""
    _require_cuda(W, V)
    d_out, d = W.shape
    k = V.shape[1]
    if M is None:
        M = torch.empty(d_out, k, dtype=W.dtype, device=W.device)
    if gram is None and with_gram:
        gram = torch.empty(k, k, dtype=torch.float32, device=W.device)
    dt = _dtype_code(W.dtype)
    nwork = int(lib().gsi_build_image_work_bytes(d, k, dt)) if tensor_cores else 0
    if nwork:
        work = torch.empty(nwork, dtype=torch.uint8, device=W.device)
        _check(lib().gsi_build_image_ex(_ptr(W), _ptr(V), _ptr(M), _ptr(gram), d, d_out, k, dt, _ptr(work),
                                        nwork, _stream(stream)))
        if workspace_status(work, stream) != 0:
            raise GsiError(5, "image build: a bounded device wait gave up")
    else:
        _check(lib().gsi_build_image(_ptr(W), _ptr(V), _ptr(M), _ptr(gram), d, d_out, k, dt, _stream(stream)))
    return M, gram


def make_map(W: torch.Tensor, V: torch.Tensor, stream=None) -> Map:
    """Upload-ready map: builds the image and the Gram on the GPU."""
    M, gram = build_image(W, V, stream=stream)
    return Map(W, V, M, gram)


def workspace_size(m: Map, T: int, path: str = "auto") -> int:
    n = ctypes.c_size_t(0)
    desc = m.desc()
    _check(lib().gsi_linear_workspace_size(ctypes.byref(desc), T, PATHS[path], ctypes.byref(n)))
    return n.value


def stack_workspace_size(maps, T: int) -> int:
    arr = (MapDesc * len(maps))(*[m.desc() for m in maps])
    n = ctypes.c_size_t(0)
    _check(lib().gsi_stack_workspace_size(arr, len(maps), T, ctypes.byref(n)))
    return n.value


def new_workspace(nbytes: int, device="cuda", stream=None) -> torch.Tensor:
    """A zero-initialised workspace of at least nbytes (256-byte aligned)."""
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    _check(lib().gsi_workspace_init(_ptr(ws), ws.numel(), _stream(stream)))
    return ws


def workspace_status(ws: torch.Tensor, stream=None) -> int:
    code = ctypes.c_uint32(0)
    st = lib().gsi_workspace_status(_ptr(ws), ctypes.byref(code), _stream(stream))
    if st not in (0, 5):
        _check(st)
    return code.value


def linear(m: Map, X: torch.Tensor, eps: float, Y=None, flags=None, rho=None, workspace=None,
           path: str = "auto", want_rho: bool = True, stream=None):
    """The gated linear map over the T tokens of X; returns (Y, flags, rho)."""
    _require_cuda(X)
    T = X.shape[0]
    dev = X.device
    if Y is None:
        Y = torch.empty(T, m.d_out, dtype=torch.float32, device=dev)
    if flags is None:
        flags = torch.empty(T, dtype=torch.uint8, device=dev)
    if rho is None and want_rho:
        rho = torch.empty(T, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(workspace_size(m, T, path), dev, stream)
    desc = m.desc()
    _check(lib().gsi_linear_ex(ctypes.byref(desc), _ptr(X), T, float(eps), _ptr(Y), _ptr(flags),
                               _ptr(rho), _ptr(workspace), workspace.numel(), PATHS[path],
                               _stream(stream)))
    return Y, flags, rho


def path_errors(m: Map, X: torch.Tensor, workspace=None, stream=None):
    """Both candidate outputs of every token and their distance.

    Returns (Y_fast, Y_slow, rho, err, ynorm): M g_t and W x_t rows, the
    residual ratios, ||Y_fast[t] - Y_slow[t]|| and ||Y_slow[t]||.
    """
    _require_cuda(X)
    T, dev = X.shape[0], X.device
    f32 = dict(dtype=torch.float32, device=dev)
    Yf, Ys = torch.empty(T, m.d_out, **f32), torch.empty(T, m.d_out, **f32)
    rho, err, ynorm = torch.empty(T, **f32), torch.empty(T, **f32), torch.empty(T, **f32)
    flags = torch.empty(T, dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = new_workspace(workspace_size(m, T), dev, stream)
    desc = m.desc()
    _check(lib().gsi_path_errors(ctypes.byref(desc), _ptr(X), T, _ptr(Yf), _ptr(Ys), _ptr(flags), _ptr(rho),
                                 _ptr(err), _ptr(ynorm), _ptr(workspace), workspace.numel(), _stream(stream)))
    return Yf, Ys, rho, err, ynorm


def eps_sweep(rho: torch.Tensor, err: torch.Tensor, ynorm: torch.Tensor, eps, tokens_per_call: int = 1,
              stream=None):
    """The gate at each threshold of `eps`; returns (n_slow, n_slow_calls, rel_err) device tensors."""
    _require_cuda(rho, err, ynorm)
    dev = rho.device
    e = torch.as_tensor(list(eps), dtype=torch.float32).to(dev)
    n = e.numel()
    n_slow = torch.empty(n, dtype=torch.int32, device=dev)
    n_calls = torch.empty(n, dtype=torch.int32, device=dev)
    rel = torch.empty(n, dtype=torch.float32, device=dev)
    _check(lib().gsi_eps_sweep(_ptr(rho), _ptr(err), _ptr(ynorm), rho.numel(), _ptr(e), n, int(tokens_per_call),
                               _ptr(n_slow), _ptr(n_calls), _ptr(rel), _stream(stream)))
    return n_slow, n_calls, rel


def basis_orthonormalize(Vt: torch.Tensor, stream=None):
    """DGKS Gram-Schmidt of the rows of Vt (k x d float32) in place; returns
    (Vt, n_reorth) with n_reorth a device int32 tensor."""
    _require_cuda(Vt)
    n = torch.zeros(1, dtype=torch.int32, device=Vt.device)
    _check(lib().gsi_basis_orthonormalize(_ptr(Vt), Vt.shape[0], Vt.shape[1], _ptr(n), _stream(stream)))
    return Vt, n


def basis_step(X: torch.Tensor, Vt: torch.Tensor, work=None, stream=None):
    """One correction step Vt <- DGKS((X^T X V)^T) on the calibration block X
    (T x d, float32 or bfloat16); returns (Vt, n_reorth)."""
    _require_cuda(X, Vt)
    T, d = X.shape
    k = Vt.shape[0]
    if work is None:
        work = new_workspace(int(lib().gsi_basis_step_work_bytes(T, d, k)), X.device, stream)
    n = torch.zeros(1, dtype=torch.int32, device=X.device)
    _check(lib().gsi_basis_step(_ptr(X), _dtype_code(X.dtype), T, d, k, _ptr(Vt), _ptr(work), work.numel(),
                                _ptr(n), _stream(stream)))
    return Vt, n


def basis_coherence(Vt_a: torch.Tensor, Vt_b: torch.Tensor, stream=None) -> torch.Tensor:
    """||Va^T Vb||_F^2 / k for two orthonormal bases held as k x d rows."""
    _require_cuda(Vt_a, Vt_b)
    k, d = Vt_a.shape
    out = torch.empty(1, dtype=torch.float32, device=Vt_a.device)
    work = torch.empty(k * k, dtype=torch.float32, device=Vt_a.device)
    _check(lib().gsi_basis_coherence(_ptr(Vt_a), _ptr(Vt_b), k, d, _ptr(out), _ptr(work), _stream(stream)))
    return out


def basis_export(Vt: torch.Tensor, dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """The basis in a map's layout: V = Vt^T (d x k, row-major) in `dtype`."""
    _require_cuda(Vt)
    k, d = Vt.shape
    V = torch.empty(d, k, dtype=dtype, device=Vt.device)
    _check(lib().gsi_basis_export(_ptr(Vt), k, d, _ptr(V), _dtype_code(dtype), _stream(stream)))
    return V


def gate(m: Map, X: torch.Tensor, eps: float, workspace=None, G=None, rho=None, flags=None,
         stream=None):
    """Projections, residual ratios and flags only; returns (G, rho, flags)."""
    _require_cuda(X)
    T = X.shape[0]
    if G is None:
        G = torch.empty(T, m.k, dtype=torch.float32, device=X.device)
    if rho is None:
        rho = torch.empty(T, dtype=torch.float32, device=X.device)
    if flags is None:
        flags = torch.empty(T, dtype=torch.uint8, device=X.device)
    if workspace is None:
        workspace = new_workspace(workspace_size(m, T, "stream"), X.device, stream)
    desc = m.desc()
    _check(lib().gsi_gate(ctypes.byref(desc), _ptr(X), T, float(eps), _ptr(G), _ptr(rho),
                          _ptr(flags), _ptr(workspace), workspace.numel(), _stream(stream)))
    return G, rho, flags


def residual_check(m: Map, X: torch.Tensor, G: torch.Tensor, rho: torch.Tensor, work=None, stream=None):
    """The gate's residual ratios checked against the explicit residual
    x - V g (a second pass over V); returns (rho_explicit, max_dev) with
    max_dev = max_t |rho_t^2 - rho_explicit_t^2| (device tensors)."""
    _require_cuda(X, G, rho)
    T = X.shape[0]
    rho_x = torch.empty(T, dtype=torch.float32, device=X.device)
    dev = torch.empty(1, dtype=torch.float32, device=X.device)
    if work is None:
        work = torch.empty(max(int(lib().gsi_residual_check_work_bytes(m.d, T)), 256), dtype=torch.uint8,
                           device=X.device)
    desc = m.desc()
    _check(lib().gsi_residual_check(ctypes.byref(desc), _ptr(X), T, _ptr(G), _ptr(rho), _ptr(rho_x), _ptr(dev),
                                    _ptr(work), work.numel(), _stream(stream)))
    return rho_x, dev


def apply(m: Map, X: torch.Tensor, G: torch.Tensor, workspace: torch.Tensor, Y=None, stream=None):
    """Fast / slow paths for the tokens of the preceding gate() on `workspace`."""
    _require_cuda(X, G)
    T = X.shape[0]
    if Y is None:
        Y = torch.empty(T, m.d_out, dtype=torch.float32, device=X.device)
    desc = m.desc()
    _check(lib().gsi_apply(ctypes.byref(desc), _ptr(X), _ptr(G), T, _ptr(Y), _ptr(workspace),
                           workspace.numel(), _stream(stream)))
    return Y


def compact(flags: torch.Tensor, stream=None):
    """Stable fast / slow index lists: returns (idx (2T int32), counts (2 int32))."""
    _require_cuda(flags)
    T = flags.shape[0]
    idx = torch.full((2 * max(T, 1),), -1, dtype=torch.int32, device=flags.device)
    counts = torch.zeros(2, dtype=torch.int32, device=flags.device)
    _check(lib().gsi_compact(_ptr(flags), T, _ptr(idx), _ptr(counts), _stream(stream)))
    return idx, counts


STACK_MODES = {"auto": 0, "per_map": 1, "persistent": 2}


def stack(maps, Xs, eps: float, Ys=None, flags=None, workspace=None, stream=None, mode: str = "auto"):
    """The gated map over a list of maps, each with its own tokens."""
    n = len(maps)
    T = Xs[0].shape[0]
    dev = Xs[0].device
    if Ys is None:
        Ys = [torch.empty(T, m.d_out, dtype=torch.float32, device=dev) for m in maps]
    if flags is None:
        flags = [torch.empty(T, dtype=torch.uint8, device=dev) for _ in maps]
    if workspace is None:
        workspace = new_workspace(stack_workspace_size(maps, T), dev, stream)
    args = stack_args(maps, Xs, Ys, flags)
    _check(lib().gsi_stack_ex(args[0], n, args[1], T, float(eps), args[2], args[3],
                              _ptr(workspace), workspace.numel(), STACK_MODES[mode], _stream(stream)))
    return Ys, flags


def stack_args(maps, Xs, Ys, flags):
    """ctypes arrays for gsi_stack (build once, reuse across calls)."""
    n = len(maps)
    vp = ctypes.c_void_p
    return ((MapDesc * n)(*[m.desc() for m in maps]),
            (vp * n)(*[x.data_ptr() for x in Xs]),
            (vp * n)(*[y.data_ptr() for y in Ys]),
            (vp * n)(*[f.data_ptr() for f in flags]))


def stack_raw(args, n, T, eps, workspace, stream=None, mode: str = "auto"):
    """gsi_stack_ex on prepared ctypes arrays (no per-call Python allocation)."""
    _check(lib().gsi_stack_ex(args[0], n, args[1], T, float(eps), args[2], args[3],
                              _ptr(workspace), workspace.numel(), STACK_MODES[mode], _stream(stream)))
