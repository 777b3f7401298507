"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the fp64 oracle on the same bf16 inputs."""
from __future__ import annotations

import numpy as np
import torch

from causal_attention_score_gb300 import synth

TOL = 1e-3  # max |gpu - oracle| <= TOL * (1 + |oracle|), on every unmasked element

NAN_BITS = 0x7FC00000
NEG_INF_BITS = 0xFF800000
POISON_BITS = 0xFFFFFFFF  # a NaN that neither mask pattern equals: catches unwritten elements


def poisoned(shape, device="cuda") -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.view(torch.int32).fill_(-1)
    return t


def f32_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32)


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str) -> None:
    gpu = gpu.astype(np.float64)
    if gpu.shape != ref.shape:
        raise AssertionError(f"{what}: shape {gpu.shape} vs {ref.shape}")
    if not np.all(np.isfinite(gpu)):
        bad = np.argwhere(~np.isfinite(gpu))[:5]
        raise AssertionError(f"{what}: non-finite GPU values at {bad.tolist()}")
    err = np.abs(gpu - ref) / (1.0 + np.abs(ref))
    worst = float(err.max()) if err.size else 0.0
    if worst > TOL:
        idx = np.unravel_index(int(err.argmax()), err.shape)
        raise AssertionError(f"{what}: max scaled error {worst:.3e} at {idx}: "
                             f"gpu {gpu[idx]!r} oracle {ref[idx]!r}")


def check_trimul_full(out_bits: np.ndarray, out_f: np.ndarray, ref: np.ndarray, mask_bits: int,
                      what: str) -> None:
    """Bit-exact mask where the oracle masks, tolerance elsewhere."""
    masked = np.isnan(ref) | np.isinf(ref)
    T = ref.shape[-1]
    upper = np.triu(np.ones((T, T), dtype=bool), k=1)
    assert np.array_equal(masked, np.broadcast_to(upper, ref.shape)), f"{what}: oracle mask shape"
    wrong = masked & (out_bits != mask_bits)
    if wrong.any():
        idx = np.argwhere(wrong)[:5].tolist()
        raise AssertionError(f"{what}: mask bits differ at {idx} "
                             f"(got {[hex(out_bits[tuple(i)]) for i in idx]})")
    assert_close(out_f[~masked], ref[~masked], what)


def trimul_case(B, T, NH, HS, seed=0, dist="normal"):
    shape = synth.TrimulShape(B=B, T=T, C=NH * HS, NH=NH)
    qkv = synth.trimul_input(shape, seed=seed, dist=dist)
    return shape, qkv
