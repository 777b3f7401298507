"""Python binding of the C ABI: argument marshalling only.

Every function checks that the tensors match what the C entry point expects
(device, dtype, contiguity, size), then passes raw pointers and the current
torch CUDA stream. All computation happens in the library's kernels.
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import CSA_MASK_NAN, CSA_MASK_NEG_INF, CSA_TRIMUL_FULL, CSA_TRIMUL_LOWER_ONLY


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, numel: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")


def _mask_bits(mask) -> int:
    if mask in ("nan", None):
        return CSA_MASK_NAN
    if mask in ("-inf", "neg_inf"):
        return CSA_MASK_NEG_INF
    return int(mask) & 0xFFFFFFFF


def trimul_forward(out: torch.Tensor, qkv: torch.Tensor, B: int, T: int, C: int, NH: int,
                   mask="nan", lower_only: bool = False, stream=None) -> None:
    """Causal scores into ``out`` (fp32, (B, NH, T, T)) from packed ``qkv``
    (bf16, (B, T, 3, NH, HS)); see trimul_forward_ex in include/csa.h."""
    _need(qkv, "qkv", torch.bfloat16, B * T * 3 * C)
    _need(out, "out", torch.float32, B * NH * T * T)
    flags = CSA_TRIMUL_LOWER_ONLY if lower_only else CSA_TRIMUL_FULL
    rc = _lib.load().trimul_forward_ex(out.data_ptr(), qkv.data_ptr(), B, T, C, NH,
                                       _mask_bits(mask), flags, _stream_ptr(stream))
    _lib.check(rc, "trimul_forward")


def trimul_forward_f32(out: torch.Tensor, qkv: torch.Tensor, B: int, T: int, C: int, NH: int,
                       mask="nan", lower_only: bool = False, stream=None) -> None:
    """Causal scores into ``out`` (fp32, (B, NH, T, T)) from packed fp32 ``qkv``
    ((B, T, 3, NH, HS), not rounded to bf16); see trimul_forward_f32 in include/csa.h."""
    _need(qkv, "qkv", torch.float32, B * T * 3 * C)
    _need(out, "out", torch.float32, B * NH * T * T)
    flags = CSA_TRIMUL_LOWER_ONLY if lower_only else CSA_TRIMUL_FULL
    rc = _lib.load().trimul_forward_f32(out.data_ptr(), qkv.data_ptr(), B, T, C, NH,
                                        _mask_bits(mask), flags, _stream_ptr(stream))
    _lib.check(rc, "trimul_forward_f32")


def dense_workspace_size(X: torch.Tensor, W: torch.Tensor, M: int, I: int, H: int) -> int:
    """Bytes of workspace ``dense_xwt_ws`` needs for these operands (0 when the rows of
    X and W can be fetched by TMA as they are); see dense_xwt_workspace_size in
    include/csa.h."""
    import ctypes
    n = ctypes.c_size_t(0)
    rc = _lib.load().dense_xwt_workspace_size(X.data_ptr(), W.data_ptr(), M, I, H,
                                               ctypes.byref(n))
    _lib.check(rc, "dense_xwt_workspace_size")
    return int(n.value)


def dense_xwt(Y: torch.Tensor, X: torch.Tensor, W: torch.Tensor, M: int, I: int, H: int,
              stream=None) -> None:
    """Y = X W^T into ``Y`` (fp32 [M, H]) from bf16 X [M, I] and W [H, I].

    Where no tensor map can describe the rows of X and W (I * 2 not a multiple of 16,
    or misaligned views), the kernel realigns them into a workspace that this binding
    takes from torch's caching allocator on the call's stream (caller memory: the
    library itself allocates nothing) and passes to dense_xwt_ws."""
    _need(X, "X", torch.bfloat16, M * I)
    _need(W, "W", torch.bfloat16, H * I)
    _need(Y, "Y", torch.float32, M * H)
    lib = _lib.load()
    nbytes = dense_workspace_size(X, W, M, I, H)
    if nbytes == 0:
        rc = lib.dense_xwt_ex(Y.data_ptr(), X.data_ptr(), W.data_ptr(), M, I, H,
                              _stream_ptr(stream))
        _lib.check(rc, "dense_xwt")
        return
    # The workspace is in use until the kernel completes on `stream`: allocated with
    # that stream current, so the caching allocator reuses it only in stream order.
    if stream is None:
        st = torch.cuda.current_stream(X.device)
    elif isinstance(stream, torch.cuda.Stream):
        st = stream
    else:
        st = torch.cuda.ExternalStream(int(stream), device=X.device)
    with torch.cuda.stream(st):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=X.device)
    rc = lib.dense_xwt_ws(Y.data_ptr(), X.data_ptr(), W.data_ptr(), M, I, H, ws.data_ptr(),
                          nbytes, int(st.cuda_stream))
    _lib.check(rc, "dense_xwt_ws")


def dense_xwt_ws(Y: torch.Tensor, X: torch.Tensor, W: torch.Tensor, M: int, I: int, H: int,
                 workspace: torch.Tensor | None, stream=None) -> None:
    """dense_xwt with a caller-provided workspace (a CUDA tensor of at least
    ``dense_workspace_size`` bytes, or None when that size is 0)."""
    _need(X, "X", torch.bfloat16, M * I)
    _need(W, "W", torch.bfloat16, H * I)
    _need(Y, "Y", torch.float32, M * H)
    ptr, nbytes = 0, 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ptr, nbytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    rc = _lib.load().dense_xwt_ws(Y.data_ptr(), X.data_ptr(), W.data_ptr(), M, I, H, ptr or None,
                                  nbytes, _stream_ptr(stream))
    _lib.check(rc, "dense_xwt_ws")


class DenseGroupedPlan:
    """dense_xwt_grouped with its arguments checked and marshalled once.

    Calling the plan launches Y[g] = X[g] W^T for every g on ``stream``; a call costs
    one C call plus a check that every tensor still has the storage it was planned
    with, instead of the full per-tensor checks (which take longer than the launch
    itself for a few dozen problems). The plan keeps references to its tensors.

    When no tensor map can describe the rows (I * 2 not a multiple of 16, or a
    misaligned view), the plan also holds the workspace dense_xwt_grouped_ws copies
    them into (torch memory, allocated once with the plan), so the batch still runs as
    one grouped launch; calls of one plan must then not overlap on the GPU.
    """

    def __init__(self, Ys, Xs, W: torch.Tensor, I: int, H: int):
        import ctypes
        if len(Ys) != len(Xs) or not Xs:
            raise ValueError("Ys and Xs must be non-empty lists of the same length")
        _need(W, "W", torch.bfloat16, H * I)
        Ms = []
        for g, (Y, X) in enumerate(zip(Ys, Xs)):
            if X.dim() != 2 or X.shape[1] != I:
                raise ValueError(f"X[{g}] must be [M, {I}]")
            M = int(X.shape[0])
            _need(X, f"X[{g}]", torch.bfloat16, M * I)
            _need(Y, f"Y[{g}]", torch.float32, M * H)
            Ms.append(M)
        n = len(Xs)
        self._tensors = [W] + list(Ys) + list(Xs)
        self._ptrs = [t.data_ptr() for t in self._tensors]
        self._y = (ctypes.c_void_p * n)(*[Y.data_ptr() for Y in Ys])
        self._x = (ctypes.c_void_p * n)(*[X.data_ptr() for X in Xs])
        self._m = (ctypes.c_int * n)(*Ms)
        self._args = (ctypes.addressof(self._y), ctypes.addressof(self._x), W.data_ptr(),
                      ctypes.addressof(self._m), n, I, H)
        nbytes = ctypes.c_size_t(0)
        _lib.check(_lib.load().dense_xwt_grouped_workspace_size(
            ctypes.addressof(self._x), W.data_ptr(), ctypes.addressof(self._m), n, I, H,
            ctypes.byref(nbytes)), "dense_xwt_grouped_workspace_size")
        self._ws = (torch.empty(nbytes.value, dtype=torch.uint8, device=W.device)
                    if nbytes.value else None)
        self._ws_args = ((self._ws.data_ptr(), nbytes.value) if self._ws is not None
                         else (None, 0))

    def __call__(self, stream=None) -> None:
        if [t.data_ptr() for t in self._tensors] != self._ptrs:
            raise ValueError("a tensor of this DenseGroupedPlan no longer has the storage it "
                             "was planned with; make a new plan")
        rc = _lib.load().dense_xwt_grouped_ws(*self._args, *self._ws_args, _stream_ptr(stream))
        _lib.check(rc, "dense_xwt_grouped")


def dense_xwt_grouped(Ys, Xs, W: torch.Tensor, I: int, H: int, stream=None) -> None:
    """Y[g] = X[g] W^T for every g, one launch per 48 problems: fp32 Y[g] [M_g, H] from
    bf16 X[g] [M_g, I] and the shared W [H, I]; see dense_xwt_grouped in include/csa.h.
    For repeated calls on the same tensors, DenseGroupedPlan checks them once."""
    DenseGroupedPlan(Ys, Xs, W, I, H)(stream)


def batch_matmul_nt(Y: torch.Tensor, X: torch.Tensor, W: torch.Tensor, batch: int, T1: int,
                    T2: int, D: int, stream=None) -> None:
    """Y[i, j, k] = sum_l X[i, j, l] W[i, k, l]: bf16 X [batch, T1, D], W [batch, T2, D]
    into fp32 Y [batch, T1, T2]."""
    _need(X, "X", torch.bfloat16, batch * T1 * D)
    _need(W, "W", torch.bfloat16, batch * T2 * D)
    _need(Y, "Y", torch.float32, batch * T1 * T2)
    rc = _lib.load().batch_matmul_nt(Y.data_ptr(), X.data_ptr(), W.data_ptr(), batch, T1, T2, D,
                                     _stream_ptr(stream))
    _lib.check(rc, "batch_matmul_nt")


def causal_softmax_forward(att: torch.Tensor, qkv: torch.Tensor, B: int, T: int, C: int, NH: int,
                           stream=None) -> None:
    """Softmax over t2 <= t of the causal scores into ``att`` (fp32, (B, NH, T, T)),
    0 above the diagonal; ``qkv`` bf16 (B, T, 3, NH, HS)."""
    _need(qkv, "qkv", torch.bfloat16, B * T * 3 * C)
    _need(att, "att", torch.float32, B * NH * T * T)
    rc = _lib.load().causal_softmax_forward(att.data_ptr(), qkv.data_ptr(), B, T, C, NH,
                                            _stream_ptr(stream))
    _lib.check(rc, "causal_softmax_forward")


def causal_softmax(qkv: torch.Tensor, stream=None) -> torch.Tensor:
    """Allocating form of causal_softmax_forward."""
    B, T, three, NH, HS = qkv.shape
    if three != 3:
        raise ValueError("qkv must have shape (B, T, 3, NH, HS)")
    att = torch.empty((B, NH, T, T), dtype=torch.float32, device=qkv.device)
    causal_softmax_forward(att, qkv, B, T, NH * HS, NH, stream=stream)
    return att


def trimul(qkv: torch.Tensor, mask="nan", lower_only: bool = False, stream=None) -> torch.Tensor:
    """Allocating form: qkv (B, T, 3, NH, HS) bf16 -> scores (B, NH, T, T) fp32."""
    B, T, three, NH, HS = qkv.shape
    if three != 3:
        raise ValueError("qkv must have shape (B, T, 3, NH, HS)")
    out = torch.empty((B, NH, T, T), dtype=torch.float32, device=qkv.device)
    trimul_forward(out, qkv, B, T, NH * HS, NH, mask=mask, lower_only=lower_only, stream=stream)
    return out


def dense(X: torch.Tensor, W: torch.Tensor, stream=None) -> torch.Tensor:
    """Allocating form: X [M, I], W [H, I] bf16 -> Y = X W^T fp32 [M, H]."""
    M, I = X.shape
    H, I2 = W.shape
    if I2 != I:
        raise ValueError("X and W disagree on I")
    Y = torch.empty((M, H), dtype=torch.float32, device=X.device)
    dense_xwt(Y, X, W, M, I, H, stream=stream)
    return Y


def get_status(stream=None) -> int:
    """Synchronise ``stream`` and return/clear the device status word (0 = ok)."""
    return int(_lib.load().csa_get_status(_stream_ptr(stream)))


def set_wait_limit_ns(ns: int) -> None:
    """Bound on every device-side wait (0 restores the default: 2 s, or the
    environment variable CSA_WAIT_LIMIT_NS)."""
    _lib.load().csa_set_wait_limit_ns(int(ns))


def get_wait_limit_ns() -> int:
    """The bound the next launch will use, in nanoseconds."""
    return int(_lib.load().csa_get_wait_limit_ns())


def debug_inject(enable: bool = True) -> None:
    _lib.load().csa_debug_inject(1 if enable else 0)


DENSE_FETCH_AUTO = 0
DENSE_FETCH_LOADERS = 1


def set_dense_fetch(mode: int) -> None:
    """Process-wide fetch mode of ``dense_xwt`` / ``dense_xwt_ws`` for rows no tensor map
    can describe: ``DENSE_FETCH_AUTO`` (rows realigned into the workspace, then TMA) or
    ``DENSE_FETCH_LOADERS`` (loader warps; the workspace unused). Same bits either way."""
    _lib.check(_lib.load().csa_set_dense_fetch(int(mode)), "csa_set_dense_fetch")


def dense_tiling(M: int, H: int, sms: int) -> tuple[int, bool]:
    """(tile width along H, CTA pairs?) that ``dense_xwt`` picks for one problem of M rows
    and H columns fetched by TMA on ``sms`` SMs; see csa_dense_tiling in include/csa.h."""
    import ctypes
    bn, pairs = ctypes.c_int(0), ctypes.c_int(0)
    _lib.check(_lib.load().csa_dense_tiling(int(M), int(H), int(sms), ctypes.byref(bn),
                                            ctypes.byref(pairs)), "csa_dense_tiling")
    return bn.value, bool(pairs.value)


def set_stream_sm_limit(stream, max_sms: int) -> None:
    """Later calls on ``stream`` (a torch stream or raw handle) size their grids for at
    most ``max_sms`` SMs, so that calls on two streams can share the GPU's SMs; 0
    removes the limit. Same bits under any limit."""
    _lib.check(_lib.load().csa_set_stream_sm_limit(_stream_ptr(stream), int(max_sms)),
               "csa_set_stream_sm_limit")


def get_stream_sm_limit(stream) -> int:
    """The SM limit set on ``stream`` (0: none)."""
    import ctypes
    v = ctypes.c_int(0)
    _lib.check(_lib.load().csa_get_stream_sm_limit(_stream_ptr(stream), ctypes.byref(v)),
               "csa_get_stream_sm_limit")
    return v.value


def version() -> str:
    return _lib.load().csa_version().decode()
