"""GB300 (sm_103a) causal attention scores and ragged dense layer.

Public API (all compute runs in libcsa_gb300.so; see include/csa.h):

* ``trimul_forward(out, qkv, B, T, C, NH, mask="nan", lower_only=False)``
* ``trimul_forward_f32(out, qkv_f32, B, T, C, NH, mask="nan", lower_only=False)``
* ``dense_xwt(Y, X, W, M, I, H)`` (``dense_xwt_ws`` with an explicit workspace,
  ``dense_workspace_size`` for its size) and ``dense_xwt_grouped(Ys, Xs, W, I, H)`` (many
  ragged X against one shared W in one launch per 48 problems; ``DenseGroupedPlan``
  checks the tensors once for repeated calls)
* ``batch_matmul_nt(Y, X, W, batch, T1, T2, D)``
* ``causal_softmax_forward(att, qkv, B, T, C, NH)``
* allocating helpers ``trimul(qkv)``, ``causal_softmax(qkv)`` and ``dense(X, W)``
* ``get_status()`` for the device watchdog word, ``set_wait_limit_ns`` /
  ``get_wait_limit_ns`` for its bound (default 2 s, or ``CSA_WAIT_LIMIT_NS``),
  ``set_dense_fetch`` for the dense layer's operand fetch mode.

The library is loaded on first use; importing this package needs no GPU.
"""
from ._lib import (CSA_ERR_ALIGN, CSA_ERR_ARCH, CSA_ERR_CHECK, CSA_ERR_CUDA, CSA_ERR_LAUNCH,
                   CSA_ERR_NULL, CSA_ERR_SHAPE, CSA_ERR_TIMEOUT, CSA_ERR_UNSUPPORTED,
                   CSA_ERR_WORKSPACE,
                   CSA_MASK_NAN, CSA_MASK_NEG_INF, CSA_OK, CsaError)
from .ops import (DENSE_FETCH_AUTO, DENSE_FETCH_LOADERS, DenseGroupedPlan, batch_matmul_nt,
                  causal_softmax, causal_softmax_forward, debug_inject, dense, dense_workspace_size,
                  dense_tiling, dense_xwt, dense_xwt_ws,
                  dense_xwt_grouped, get_status, get_stream_sm_limit, get_wait_limit_ns,
                  set_dense_fetch, set_stream_sm_limit, set_wait_limit_ns, trimul, trimul_forward,
                  trimul_forward_f32, version)

__all__ = [
    "trimul_forward", "trimul_forward_f32", "dense_xwt", "dense_xwt_ws", "dense_workspace_size",
    "dense_xwt_grouped", "DenseGroupedPlan",
    "batch_matmul_nt", "causal_softmax_forward", "causal_softmax", "trimul", "dense", "get_status",
    "set_wait_limit_ns", "get_wait_limit_ns", "debug_inject", "set_dense_fetch",
    "set_stream_sm_limit", "get_stream_sm_limit", "dense_tiling",
    "DENSE_FETCH_AUTO", "DENSE_FETCH_LOADERS", "version", "CsaError", "CSA_OK", "CSA_ERR_NULL",
    "CSA_ERR_SHAPE",
    "CSA_ERR_ALIGN", "CSA_ERR_UNSUPPORTED", "CSA_ERR_ARCH", "CSA_ERR_LAUNCH", "CSA_ERR_TIMEOUT",
    "CSA_ERR_CUDA", "CSA_ERR_CHECK", "CSA_ERR_WORKSPACE", "CSA_MASK_NAN", "CSA_MASK_NEG_INF",
]
