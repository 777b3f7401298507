"""fp64 CPU oracle (test infrastructure).

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / reference leg may import this package. The product path
(the CUDA library and its Python binding) never does, and shares no code with
it: the oracle is a separate plain-C file compiled with gcc.

The C source (``csa_oracle.c``) states, per function, the passage of the
pages it follows:

* ``trimul`` / ``trimul_rows``: the CPU referee ``trimul_cpu`` of
  "llm.c dev/cuda/trimat_forward.cu" (Chapter I).
* ``trimul_f32`` / ``trimul_f32_rows``: the same referee over its own fp32
  input type (no bf16 rounding of the inputs).
* ``dense`` / ``dense_rows``: the dense workload ``Y = X W^T`` of
  "DietCode tests/codegen/test_1_local_padding.py" (test_local_padding
  docstring).
* ``causal_softmax`` / ``causal_softmax_rows``: the two-pass row softmax of the
  "Smallem" article 5 (kernels-gpu) over each causal score row (t2 <= t), 0 above.
* ``bmm_nt``: the batched NT workload of the same file (test_local_padding_ii
  docstring), ``Y[i, j, k] = sum_l X[i, j, l] W[i, k, l]``.

Inputs are bf16 tensors passed as their raw 16-bit patterns (numpy uint16),
or numpy float32 for the fp32-input functions; outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "csa_oracle.c")
LIBPATH = os.path.join(_HERE, "_build", "libcsa_oracle.so")

MASK_NAN = 0
MASK_NEG_INF = 1

_lock = threading.Lock()


def compile_oracle(source: str = SOURCE, out: str = LIBPATH, force: bool = False) -> str:
    """Compile the C oracle into a shared library (gcc, -O2, OpenMP, no fast-math)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(source):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes view of one compiled oracle library (the default one, or a
    deliberately mutated copy that the mutation tests build)."""

    def __init__(self, libpath: str):
        self.lib = ctypes.CDLL(libpath)
        i64 = ctypes.c_int64
        dp = ctypes.POINTER(ctypes.c_double)
        up = ctypes.POINTER(ctypes.c_uint16)
        lp = ctypes.POINTER(ctypes.c_int64)
        self.lib.oracle_trimul.argtypes = [dp, up, i64, i64, i64, i64, ctypes.c_int]
        self.lib.oracle_trimul_rows.argtypes = [dp, up, i64, i64, i64, i64, lp, i64, ctypes.c_int]
        self.lib.oracle_dense.argtypes = [dp, up, up, i64, i64, i64]
        self.lib.oracle_dense_rows.argtypes = [dp, up, up, i64, i64, i64, lp, i64]
        self.lib.oracle_bmm_nt.argtypes = [dp, up, up, i64, i64, i64, i64]
        self.lib.oracle_causal_softmax.argtypes = [dp, up, i64, i64, i64, i64]
        self.lib.oracle_causal_softmax_rows.argtypes = [dp, up, i64, i64, i64, i64, lp, i64]
        fp = ctypes.POINTER(ctypes.c_float)
        self.lib.oracle_trimul_f32.argtypes = [dp, fp, i64, i64, i64, i64, ctypes.c_int]
        self.lib.oracle_trimul_f32_rows.argtypes = [dp, fp, i64, i64, i64, i64, lp, i64, ctypes.c_int]
        for f in ("oracle_trimul", "oracle_trimul_rows", "oracle_dense", "oracle_dense_rows",
                  "oracle_bmm_nt", "oracle_causal_softmax", "oracle_causal_softmax_rows",
                  "oracle_trimul_f32", "oracle_trimul_f32_rows", "oracle_num_threads"):
            getattr(self.lib, f).restype = ctypes.c_int
        self.lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        self.lib.oracle_set_num_threads.restype = None

    # -- threads -----------------------------------------------------------
    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.lib.oracle_set_num_threads(int(n))

    # -- causal score product ---------------------------------------------
    def trimul(self, qkv_u16: np.ndarray, B: int, T: int, C: int, NH: int,
               mask: int = MASK_NAN) -> np.ndarray:
        """Scores (B, NH, T, T) float64 of the packed (B, T, 3, NH, HS) input."""
        q = np.ascontiguousarray(qkv_u16, dtype=np.uint16)
        if q.size != B * T * 3 * C:
            raise ValueError("qkv size does not match (B, T, 3, C)")
        out = np.empty((B, NH, T, T), dtype=np.float64)
        rc = self.lib.oracle_trimul(_ptr(out, ctypes.c_double), _ptr(q, ctypes.c_uint16),
                                    B, T, C, NH, mask)
        if rc != 0:
            raise ValueError(f"oracle_trimul rejected the shape (rc={rc})")
        return out

    def trimul_rows(self, qkv_u16: np.ndarray, B: int, T: int, C: int, NH: int,
                    bht: np.ndarray, mask: int = MASK_NAN) -> np.ndarray:
        """Rows out[b, h, t, :] for each (b, h, t) in bht (n x 3); returns n x T."""
        q = np.ascontiguousarray(qkv_u16, dtype=np.uint16)
        idx = np.ascontiguousarray(bht, dtype=np.int64).reshape(-1, 3)
        out = np.empty((idx.shape[0], T), dtype=np.float64)
        rc = self.lib.oracle_trimul_rows(_ptr(out, ctypes.c_double), _ptr(q, ctypes.c_uint16),
                                         B, T, C, NH, _ptr(idx, ctypes.c_int64),
                                         idx.shape[0], mask)
        if rc != 0:
            raise ValueError(f"oracle_trimul_rows rejected the arguments (rc={rc})")
        return out

    # -- causal score product, fp32 inputs -------------------------------
    def trimul_f32(self, qkv_f32: np.ndarray, B: int, T: int, C: int, NH: int,
                   mask: int = MASK_NAN) -> np.ndarray:
        """Scores (B, NH, T, T) float64 of the packed (B, T, 3, NH, HS) fp32 input."""
        q = np.ascontiguousarray(qkv_f32, dtype=np.float32)
        if q.size != B * T * 3 * C:
            raise ValueError("qkv size does not match (B, T, 3, C)")
        out = np.empty((B, NH, T, T), dtype=np.float64)
        rc = self.lib.oracle_trimul_f32(_ptr(out, ctypes.c_double), _ptr(q, ctypes.c_float),
                                        B, T, C, NH, mask)
        if rc != 0:
            raise ValueError(f"oracle_trimul_f32 rejected the shape (rc={rc})")
        return out

    def trimul_f32_rows(self, qkv_f32: np.ndarray, B: int, T: int, C: int, NH: int,
                        bht: np.ndarray, mask: int = MASK_NAN) -> np.ndarray:
        """Rows out[b, h, t, :] of the fp32-input scores for each (b, h, t) in bht."""
        q = np.ascontiguousarray(qkv_f32, dtype=np.float32)
        idx = np.ascontiguousarray(bht, dtype=np.int64).reshape(-1, 3)
        out = np.empty((idx.shape[0], T), dtype=np.float64)
        rc = self.lib.oracle_trimul_f32_rows(_ptr(out, ctypes.c_double), _ptr(q, ctypes.c_float),
                                             B, T, C, NH, _ptr(idx, ctypes.c_int64),
                                             idx.shape[0], mask)
        if rc != 0:
            raise ValueError(f"oracle_trimul_f32_rows rejected the arguments (rc={rc})")
        return out

    # -- dense layer -------------------------------------------------------
    def dense(self, X_u16: np.ndarray, W_u16: np.ndarray, M: int, I: int, H: int) -> np.ndarray:
        """Y = X W^T as (M, H) float64."""
        x = np.ascontiguousarray(X_u16, dtype=np.uint16)
        w = np.ascontiguousarray(W_u16, dtype=np.uint16)
        if x.size != M * I or w.size != H * I:
            raise ValueError("X / W sizes do not match (M, I) / (H, I)")
        Y = np.empty((M, H), dtype=np.float64)
        rc = self.lib.oracle_dense(_ptr(Y, ctypes.c_double), _ptr(x, ctypes.c_uint16),
                                   _ptr(w, ctypes.c_uint16), M, I, H)
        if rc != 0:
            raise ValueError(f"oracle_dense rejected the shape (rc={rc})")
        return Y

    def dense_rows(self, X_u16: np.ndarray, W_u16: np.ndarray, M: int, I: int, H: int,
                   rows: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(X_u16, dtype=np.uint16)
        w = np.ascontiguousarray(W_u16, dtype=np.uint16)
        r = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
        Y = np.empty((r.shape[0], H), dtype=np.float64)
        rc = self.lib.oracle_dense_rows(_ptr(Y, ctypes.c_double), _ptr(x, ctypes.c_uint16),
                                        _ptr(w, ctypes.c_uint16), M, I, H,
                                        _ptr(r, ctypes.c_int64), r.shape[0])
        if rc != 0:
            raise ValueError(f"oracle_dense_rows rejected the arguments (rc={rc})")
        return Y


    # -- batched NT product -----------------------------------------------
    def bmm_nt(self, X_u16: np.ndarray, W_u16: np.ndarray, batch: int, T1: int, T2: int,
               D: int) -> np.ndarray:
        """Y[i, j, k] = sum_l X[i, j, l] W[i, k, l] as (batch, T1, T2) float64."""
        x = np.ascontiguousarray(X_u16, dtype=np.uint16)
        w = np.ascontiguousarray(W_u16, dtype=np.uint16)
        if x.size != batch * T1 * D or w.size != batch * T2 * D:
            raise ValueError("X / W sizes do not match (batch, T1, D) / (batch, T2, D)")
        Y = np.empty((batch, T1, T2), dtype=np.float64)
        rc = self.lib.oracle_bmm_nt(_ptr(Y, ctypes.c_double), _ptr(x, ctypes.c_uint16),
                                    _ptr(w, ctypes.c_uint16), batch, T1, T2, D)
        if rc != 0:
            raise ValueError(f"oracle_bmm_nt rejected the shape (rc={rc})")
        return Y


    # -- causal softmax ---------------------------------------------------
    def causal_softmax(self, qkv_u16: np.ndarray, B: int, T: int, C: int, NH: int) -> np.ndarray:
        """Softmax over t2 <= t of each causal score row, 0 above; (B, NH, T, T) float64."""
        q = np.ascontiguousarray(qkv_u16, dtype=np.uint16)
        if q.size != B * T * 3 * C:
            raise ValueError("qkv size does not match (B, T, 3, C)")
        out = np.empty((B, NH, T, T), dtype=np.float64)
        rc = self.lib.oracle_causal_softmax(_ptr(out, ctypes.c_double), _ptr(q, ctypes.c_uint16),
                                            B, T, C, NH)
        if rc != 0:
            raise ValueError(f"oracle_causal_softmax rejected the shape (rc={rc})")
        return out

    def causal_softmax_rows(self, qkv_u16: np.ndarray, B: int, T: int, C: int, NH: int,
                            bht: np.ndarray) -> np.ndarray:
        q = np.ascontiguousarray(qkv_u16, dtype=np.uint16)
        idx = np.ascontiguousarray(bht, dtype=np.int64).reshape(-1, 3)
        out = np.empty((idx.shape[0], T), dtype=np.float64)
        rc = self.lib.oracle_causal_softmax_rows(_ptr(out, ctypes.c_double),
                                                 _ptr(q, ctypes.c_uint16), B, T, C, NH,
                                                 _ptr(idx, ctypes.c_int64), idx.shape[0])
        if rc != 0:
            raise ValueError(f"oracle_causal_softmax_rows rejected the arguments (rc={rc})")
        return out


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from ``csa_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(compile_oracle())
        return _default
