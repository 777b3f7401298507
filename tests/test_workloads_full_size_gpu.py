"""The measured workloads that other files check only at small sizes, at their full
sizes and in the launch configuration the benchmark times: every element checked
for what it must be (untouched, masked, zero, finite), sampled rows against the
oracle (GPU)."""
import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import synth
from gpu_util import (POISON_BITS, assert_close, assert_softmax_close, f32_bits,
                      softmax_abs_scores, softmax_rel_bound)

pytestmark = pytest.mark.gpu

F32_REL = 2.0 ** -15  # the 3 x tf32 bound per score, relative to sum |q_i k_i| / sqrt(HS)


def _rows(shape, seed, per_bh=2):
    rng = np.random.default_rng(seed)
    T = shape.T
    return np.array([(b, h, int(t)) for b in range(shape.B) for h in range(shape.NH)
                     for t in sorted({0, T - 1, T // 2, *rng.integers(0, T, size=per_bh).tolist()})],
                    dtype=np.int64)


@pytest.mark.parametrize("shape", [synth.TRIMUL_GPT2, synth.TRIMUL_LONG], ids=["gpt2", "long"])
def test_lower_only_full_size(oracle_lib, shape):
    qkv = synth.trimul_input(shape, seed=0, dist="normal")
    out = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")
    out.view(torch.int32).fill_(-1)
    csa.trimul_forward(out, qkv.cuda(), shape.B, shape.T, shape.C, shape.NH, lower_only=True)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    T = shape.T
    upper = torch.triu(torch.ones((T, T), dtype=torch.bool, device="cuda"), diagonal=1)
    for b in range(shape.B):
        for h in range(shape.NH):
            s = out[b, h]
            assert bool(torch.all(s.view(torch.int32)[upper] == -1)), (b, h)  # untouched
            assert bool(torch.all(torch.isfinite(s[~upper]))), (b, h)
    bht = _rows(shape, seed=3)
    ref = oracle_lib.trimul_rows(synth.bf16_bits(qkv).reshape(-1), shape.B, T, shape.C,
                                 shape.NH, bht, 0)
    idx = torch.from_numpy(bht).cuda()
    got = out[idx[:, 0], idx[:, 1], idx[:, 2]]
    gbits, gf = f32_bits(got), got.cpu().numpy()
    for i, (b, h, t) in enumerate(bht):
        assert np.all(gbits[i, t + 1:] == POISON_BITS), (b, h, t)
        assert_close(gf[i, :t + 1], ref[i, :t + 1], f"lower-only {shape} row {(b, h, t)}")


def test_softmax_long_context_full_size(oracle_lib):
    s = synth.TRIMUL_LONG
    qkv = synth.trimul_input(s, seed=0, dist="normal")
    att = torch.empty(s.out_shape, dtype=torch.float32, device="cuda")
    csa.causal_softmax_forward(att, qkv.cuda(), s.B, s.T, s.C, s.NH)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    T = s.T
    upper = torch.triu(torch.ones((T, T), dtype=torch.bool, device="cuda"), diagonal=1)
    for b in range(s.B):
        for h in range(s.NH):
            p = att[b, h]
            assert bool(torch.all(p[upper] == 0)), (b, h)
            assert float((p.sum(dim=-1) - 1).abs().max()) <= 1e-4, (b, h)
    bht = _rows(s, seed=4)
    ref = oracle_lib.causal_softmax_rows(synth.bf16_bits(qkv).reshape(-1), s.B, T, s.C, s.NH, bht)
    idx = torch.from_numpy(bht).cuda()
    got = att[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy()
    assert_close(got, ref, "long-context softmax rows")
    rel = softmax_rel_bound(softmax_abs_scores(oracle_lib, qkv, s.B, T, s.C, s.NH, bht),
                            bht[:, 2], s.HS)
    rel = np.where(np.arange(T)[None, :] > bht[:, 2:3], np.inf, rel)
    assert_softmax_close(got, ref, rel, "long-context softmax rows (relative bound)")


def test_trimul_f32_long_context_full_size(oracle_lib):
    shape = synth.TRIMUL_LONG
    qkv = synth.trimul_input_f32(shape, seed=0, dist="uniform")
    out = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")
    csa.trimul_forward_f32(out, qkv.cuda(), shape.B, shape.T, shape.C, shape.NH)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    T = shape.T
    upper = torch.triu(torch.ones((T, T), dtype=torch.bool, device="cuda"), diagonal=1)
    for b in range(shape.B):
        for h in range(shape.NH):
            s = out[b, h]
            assert bool(torch.all(s.view(torch.int32)[upper] == 0x7FC00000)), (b, h)
            assert bool(torch.all(torch.isfinite(s[~upper]))), (b, h)
    bht = _rows(shape, seed=6)
    x = qkv.numpy().reshape(-1)
    ref = oracle_lib.trimul_f32_rows(x, shape.B, T, shape.C, shape.NH, bht, 0)
    ref_abs = oracle_lib.trimul_f32_rows(np.abs(x), shape.B, T, shape.C, shape.NH, bht, 0)
    idx = torch.from_numpy(bht).cuda()
    got = out[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy().astype(np.float64)
    for i, (b, h, t) in enumerate(bht):
        err = np.abs(got[i, :t + 1] - ref[i, :t + 1])
        assert float(err.max()) <= 1e-3, (b, h, t, float(err.max()))
        assert np.all(err <= F32_REL * ref_abs[i, :t + 1] + 1e-30), (b, h, t)
