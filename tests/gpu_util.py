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


# ----------------------------------------------------------- softmax bound --
#
# Per-probability bound of the fused causal softmax, from its arithmetic. With
# a(t, u) = sum_d |q_{t,d} k_{u,d}| / sqrt(HS) (the oracle's score of |Q| and |K|)
# and A(t) = max_{u <= t} a(t, u):
#  - each score carries at most (HS + 4) * 2^-24 * a(t, u) of absolute error (fp32
#    accumulation of HS exact bf16 products, the scale's and the log2(e) factor's
#    roundings); log p = s_u - logsumexp(s) moves by at most the error of s_u plus
#    the largest error in the row, so p moves by that much relatively;
#  - the fp32 sum of the t + 1 exponentials: (t + 1) * 2^-24;
#  - the exponent argument (x - m) - log2 l, of magnitude < 160 where p is not
#    flushed: 160 * 2^-24;
#  - the running-maximum rescales of l, one per 32 columns at most: 2^-22 each;
#  - the approximate exp2 / log2 instructions (a few units of 2^-22 each): 2^-20.
# Below 2^-125 the exp2 result may be flushed to zero: an absolute floor.
SOFTMAX_FLOOR = 2.0 ** -125


def softmax_rel_bound(abs_rows: np.ndarray, t: np.ndarray, HS: int) -> np.ndarray:
    """Relative bound per probability for rows of a(t, u) (NaN above the diagonal);
    `t` gives each row's query index (broadcast against abs_rows[..., 0])."""
    a = np.where(np.isnan(abs_rows), 0.0, abs_rows)
    A = a.max(axis=-1, keepdims=True)
    t = np.asarray(t, dtype=np.float64)[..., None]
    u = 2.0 ** -24
    return ((HS + 4) * u * (a + A) + (t + 1 + 160) * u + np.ceil((t + 1) / 32) * 2.0 ** -22
            + 2.0 ** -20)


def assert_softmax_close(got: np.ndarray, ref: np.ndarray, rel: np.ndarray, what: str) -> None:
    """|got - ref| <= ref * rel + 2^-125 on every entry at or below the diagonal (where
    rel is finite); the caller checks the zeros above it bit-exactly."""
    got = got.astype(np.float64)
    live = np.isfinite(rel) & ~np.isnan(ref)
    err = np.abs(got - ref)
    bound = np.where(live, np.where(live, ref, 0.0) * np.where(live, rel, 0.0), 0.0) + SOFTMAX_FLOOR
    bad = live & ~(err <= bound)
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: probability {got[idx]!r} vs oracle {ref[idx]!r} at {idx}: "
                             f"error {err[idx]:.3e} above the bound {bound[idx]:.3e}")


def softmax_abs_scores(oracle_lib, qkv: torch.Tensor, B: int, T: int, C: int, NH: int,
                       bht: np.ndarray | None = None) -> np.ndarray:
    """a(t, u) from the oracle's score of |Q| and |K| (bf16 magnitudes are exact):
    (B, NH, T, T), or the rows of bht (n x T); NaN above the diagonal."""
    bits = synth.bf16_bits(qkv).reshape(-1) & np.uint16(0x7FFF)
    if bht is None:
        return oracle_lib.trimul(bits, B, T, C, NH)
    return oracle_lib.trimul_rows(bits, B, T, C, NH, bht)
