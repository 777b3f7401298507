"""Seeded synthetic inputs for the two products.

This module is shared by the tests, the benchmark and the oracle checks, and
holds none of the products' arithmetic: it only draws random numbers and
rounds them to bf16 (round-to-nearest-even, done by torch on the CPU). Both
sides of every comparison consume the same bf16 tensor.

Workload shapes follow the pages:

* the score product's input is the packed QKV tensor (B, T, 3, NH, HS) of
  "llm.c dev/cuda/trimat_forward.cu" (its ``main`` uses B=8, T=1024, C=768,
  NH=12);
* the dense layer uses X [B*T, I], W [H, I] of
  "DietCode tests/codegen/test_1_local_padding.py" (B, T, I = 16, 60, 770).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a CPU bf16 tensor as a numpy uint16 array."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def uniform_bf16(shape, seed: int, lo: float = -1.0, hi: float = 1.0,
                 generator: torch.Generator | None = None) -> torch.Tensor:
    """fp32 iid uniform[lo, hi) from ``seed`` (or a running generator), rounded to bf16."""
    g = generator if generator is not None else torch.Generator().manual_seed(seed)
    x = torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo
    return x.to(torch.bfloat16)


def normal_bf16(shape, seed: int) -> torch.Tensor:
    """fp32 iid N(0, 1) from ``seed``, rounded to bf16."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


@dataclass(frozen=True)
class TrimulShape:
    B: int
    T: int
    C: int
    NH: int

    @property
    def HS(self) -> int:
        return self.C // self.NH

    @property
    def qkv_shape(self):
        return (self.B, self.T, 3, self.NH, self.HS)

    @property
    def out_shape(self):
        return (self.B, self.NH, self.T, self.T)


@dataclass(frozen=True)
class DenseShape:
    M: int
    I: int
    H: int


# The pages' workloads at the sizes this library is measured on.
TRIMUL_TINY = TrimulShape(B=1, T=64, C=128, NH=2)
TRIMUL_GPT2 = TrimulShape(B=8, T=1024, C=768, NH=12)
TRIMUL_LONG = TrimulShape(B=2, T=4096, C=2048, NH=16)
DENSE_RAGGED = DenseShape(M=16 * 60, I=770, H=768)
DENSE_SWEEP_I = 768
DENSE_SWEEP_H = 3072
DENSE_SWEEP_CALLS = 32
DENSE_SWEEP_BATCH = 16


def trimul_input(shape: TrimulShape, seed: int = 0, dist: str = "normal") -> torch.Tensor:
    """Packed QKV (B, T, 3, NH, HS) bf16 on the CPU.

    dist="uniform": iid uniform[-1, 1] (the tiny case); "normal": iid N(0, 1).
    """
    if dist == "uniform":
        return uniform_bf16(shape.qkv_shape, seed)
    if dist == "normal":
        return normal_bf16(shape.qkv_shape, seed)
    raise ValueError(dist)


def trimul_input_f32(shape: TrimulShape, seed: int = 0, dist: str = "uniform") -> torch.Tensor:
    """Packed QKV (B, T, 3, NH, HS) fp32 on the CPU, not rounded to bf16.

    dist="uniform": iid uniform[-1, 1] (what the page's ``main`` fills its fp32
    input with); "normal": iid N(0, 1).
    """
    g = torch.Generator().manual_seed(seed)
    if dist == "uniform":
        return torch.rand(shape.qkv_shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape.qkv_shape, generator=g, dtype=torch.float32)
    raise ValueError(dist)


def dense_input(shape: DenseShape, seed: int = 0):
    """(X [M, I], W [H, I]) bf16 iid uniform[-1, 1]; X is drawn first, then W,
    from one generator seeded with ``seed``."""
    g = torch.Generator().manual_seed(seed)
    X = uniform_bf16((shape.M, shape.I), seed, generator=g)
    W = uniform_bf16((shape.H, shape.I), seed, generator=g)
    return X, W


def dense_sweep_lengths(seed: int = 0, calls: int = DENSE_SWEEP_CALLS):
    """Sequence lengths T_i ~ U{1..128} of the dynamic-shape sweep (M_i = 16 * T_i)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(1, 129, (calls,), generator=g).tolist()


def dense_sweep_inputs(seed: int = 0):
    """The sweep: W [3072, 768] from seed 1, X_i [16*T_i, 768] from seed 1000+i."""
    W = uniform_bf16((DENSE_SWEEP_H, DENSE_SWEEP_I), 1)
    xs = [uniform_bf16((DENSE_SWEEP_BATCH * t, DENSE_SWEEP_I), 1000 + i)
          for i, t in enumerate(dense_sweep_lengths(seed))]
    return xs, W


@dataclass(frozen=True)
class BmmShape:
    batch: int
    T1: int
    T2: int
    D: int


# "DietCode ... test_local_padding_ii": B, T, H, NH = 16, 120, 768, 12 -> batch
# B*NH = 192, T = 120, D = H/NH = 64.
BMM_NT_RAGGED = BmmShape(batch=16 * 12, T1=120, T2=120, D=64)


def bmm_input(shape: BmmShape, seed: int = 0):
    """(X [batch, T1, D], W [batch, T2, D]) bf16 iid uniform[-1, 1]; X first, one
    generator seeded with ``seed``."""
    g = torch.Generator().manual_seed(seed)
    X = uniform_bf16((shape.batch, shape.T1, shape.D), seed, generator=g)
    W = uniform_bf16((shape.batch, shape.T2, shape.D), seed, generator=g)
    return X, W
