"""Parity of the fused causal softmax against the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import synth
from gpu_util import (assert_close, assert_softmax_close, f32_bits, poisoned,
                      softmax_abs_scores, softmax_rel_bound, trimul_case)

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 64, 2, 64),
    (2, 1, 1, 64),
    (1, 63, 2, 64),
    (1, 129, 2, 64),
    (2, 300, 3, 64),
    (1, 256, 2, 128),
    (1, 100, 1, 72),
    (1, 40, 2, 8),
    (3, 520, 1, 32),
]


def _check(att: torch.Tensor, ref: np.ndarray, what: str, abs_scores=None, HS=None) -> None:
    """Zeros above the diagonal bit-exactly; the benchmark spec's tolerance; rows summing to
    1; and, given the row's |q||k| scores, each probability within its relative bound
    (which, unlike 1e-3 * (1 + p), holds small probabilities to their own scale)."""
    T = ref.shape[-1]
    upper = np.triu(np.ones((T, T), dtype=bool), k=1)
    bits = f32_bits(att)
    assert np.all(bits[..., upper] == 0), f"{what}: nonzero above the diagonal"
    got = att.cpu().numpy()
    assert_close(got[..., ~upper], ref[..., ~upper], what)
    assert np.max(np.abs(got.sum(axis=-1) - 1.0)) <= 1e-4, f"{what}: rows do not sum to 1"
    if abs_scores is not None:
        rel = softmax_rel_bound(abs_scores, np.arange(T), HS)
        rel = np.where(np.broadcast_to(upper, rel.shape), np.inf, rel)
        assert_softmax_close(got, ref, rel, what + " (relative bound)")


@pytest.mark.parametrize("B,T,NH,HS", SHAPES)
def test_softmax_parity(oracle_lib, B, T, NH, HS):
    shape, qkv = trimul_case(B, T, NH, HS, seed=B * 7 + T + HS)
    ref = oracle_lib.causal_softmax(synth.bf16_bits(qkv).reshape(-1), B, T, shape.C, NH)
    att = poisoned(shape.out_shape)
    csa.causal_softmax_forward(att, qkv.cuda(), B, T, shape.C, NH)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    _check(att, ref, f"softmax{(B, T, NH, HS)}",
           softmax_abs_scores(oracle_lib, qkv, B, T, shape.C, NH), HS)


def test_softmax_large_scores_stay_finite(oracle_lib):
    """Scores of several hundred (exp would overflow without subtracting the row max)."""
    B, T, NH, HS = 1, 200, 2, 16
    g = torch.Generator().manual_seed(3)
    qkv = (torch.randn((B, T, 3, NH, HS), generator=g) * 12).to(torch.bfloat16)
    ref = oracle_lib.causal_softmax(synth.bf16_bits(qkv).reshape(-1), B, T, NH * HS, NH)
    scores = oracle_lib.trimul(synth.bf16_bits(qkv).reshape(-1), B, T, NH * HS, NH, 0)
    assert np.nanmax(np.abs(scores)) > 200
    att = csa.causal_softmax(qkv.cuda())
    torch.cuda.synchronize()
    _check(att, ref, "large scores", softmax_abs_scores(oracle_lib, qkv, B, T, NH * HS, NH), HS)


def test_softmax_gpt2_full_size_sampled_rows(oracle_lib):
    s = synth.TRIMUL_GPT2
    qkv = synth.trimul_input(s, seed=0, dist="normal")
    att = torch.empty(s.out_shape, dtype=torch.float32, device="cuda")
    csa.causal_softmax_forward(att, qkv.cuda(), s.B, s.T, s.C, s.NH)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    T = s.T
    rng = np.random.default_rng(1)
    bht = np.array([(b, h, t) for b in range(s.B) for h in range(s.NH)
                    for t in sorted({0, T - 1, int(rng.integers(0, T))})], dtype=np.int64)
    ref = oracle_lib.causal_softmax_rows(synth.bf16_bits(qkv).reshape(-1), s.B, T, s.C, s.NH, bht)
    idx = torch.from_numpy(bht).cuda()
    got = att[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy()
    assert_close(got, ref, "GPT-2 softmax rows")
    rel = softmax_rel_bound(softmax_abs_scores(oracle_lib, qkv, s.B, T, s.C, s.NH, bht),
                            bht[:, 2], s.HS)
    rel = np.where(np.arange(T)[None, :] > bht[:, 2:3], np.inf, rel)
    assert_softmax_close(got, ref, rel, "GPT-2 softmax rows (relative bound)")
    sums = att.sum(dim=-1)
    assert float((sums - 1).abs().max()) <= 1e-4
    upper = torch.triu(torch.ones((T, T), dtype=torch.bool, device="cuda"), diagonal=1)
    assert bool(torch.all(att[:, :, upper] == 0))
