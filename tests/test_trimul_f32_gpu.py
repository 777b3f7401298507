"""Parity of the fp32-input causal score product (3 x tf32 on tcgen05) against the
fp64 oracle over the same fp32 inputs (GPU)."""
import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import synth
from gpu_util import (NAN_BITS, NEG_INF_BITS, POISON_BITS, check_trimul_full, f32_bits,
                      poisoned)

pytestmark = pytest.mark.gpu

# Three tf32 products per input pair leave, per product, a relative error of a
# few units of 2^-20 (lo's tf32 rounding, the dropped lo.lo term); fp32
# accumulation over HS terms adds up to HS * 2^-24. Both are bounded by a
# multiple of sum_i |q_i k_i| / sqrt(HS), which the oracle computes as the score
# of |Q| and |K|. 2^-15 of it is far below what one tf32 product would leave
# (2^-10 of it) and above the 3 x tf32 error with room to spare.
F32_REL = 2.0 ** -15

SHAPES = [
    (1, 64, 2, 64),
    (2, 1, 1, 64),
    (1, 63, 2, 64),
    (1, 129, 2, 64),
    (2, 200, 3, 64),
    (1, 300, 2, 128),
    (1, 100, 1, 36),
    (1, 40, 2, 4),
    (1, 97, 2, 20),
    (1, 70, 1, 256),
    (3, 384, 1, 32),
]


def _case(B, T, NH, HS, seed, dist="normal"):
    shape = synth.TrimulShape(B=B, T=T, C=NH * HS, NH=NH)
    return shape, synth.trimul_input_f32(shape, seed=seed, dist=dist)


def _abs_scores(oracle_lib, qkv, shape):
    """sum_i |q_i k_i| / sqrt(HS) per score (the oracle's score of |Q| and |K|)."""
    return oracle_lib.trimul_f32(np.abs(qkv.numpy()).reshape(-1), shape.B, shape.T, shape.C,
                                 shape.NH, 0)


def _check_f32_bound(got, ref, scale_abs, what):
    lower = ~np.isnan(ref)
    err = np.abs(got[lower].astype(np.float64) - ref[lower])
    bound = F32_REL * scale_abs[lower] + 1e-30
    worst = float((err / bound).max()) if err.size else 0.0
    assert worst <= 1.0, f"{what}: error {worst:.2f}x the 3xtf32 bound"


@pytest.mark.parametrize("B,T,NH,HS", SHAPES)
def test_trimul_f32_parity(oracle_lib, B, T, NH, HS):
    shape, qkv = _case(B, T, NH, HS, seed=B * 1000 + T * 10 + NH)
    ref = oracle_lib.trimul_f32(qkv.numpy().reshape(-1), B, T, shape.C, NH, 0)
    out = poisoned(shape.out_shape)
    csa.trimul_forward_f32(out, qkv.cuda(), B, T, shape.C, NH)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    got = out.cpu().numpy()
    check_trimul_full(f32_bits(out), got, ref, NAN_BITS, f"trimul_f32{(B, T, NH, HS)}")
    _check_f32_bound(got, ref, _abs_scores(oracle_lib, qkv, shape), f"f32 bound {(B, T, NH, HS)}")


@pytest.mark.parametrize("T", [64, 250])
def test_trimul_f32_neg_inf_and_lower_only(oracle_lib, T):
    shape, qkv = _case(2, T, 2, 64, seed=T)
    ref = oracle_lib.trimul_f32(qkv.numpy().reshape(-1), 2, T, shape.C, 2, 1)
    out = poisoned(shape.out_shape)
    csa.trimul_forward_f32(out, qkv.cuda(), 2, T, shape.C, 2, mask="-inf")
    torch.cuda.synchronize()
    check_trimul_full(f32_bits(out), out.cpu().numpy(), ref, NEG_INF_BITS, f"f32 -inf T={T}")
    out2 = poisoned(shape.out_shape)
    csa.trimul_forward_f32(out2, qkv.cuda(), 2, T, shape.C, 2, lower_only=True)
    torch.cuda.synchronize()
    bits = f32_bits(out2)
    upper = np.triu(np.ones((T, T), dtype=bool), k=1)
    assert np.all(bits[..., upper] == POISON_BITS)
    assert np.array_equal(bits[..., ~upper], f32_bits(out)[..., ~upper])


@pytest.mark.parametrize("B,T,NH,HS", [(1, 256, 2, 64), (2, 131, 1, 16), (1, 64, 1, 256)])
def test_trimul_f32_integer_inputs_bit_exact(oracle_lib, B, T, NH, HS):
    """Small integers are tf32 values (lo = 0): every product and partial sum is exact
    and 1/sqrt(HS) is a power of two, so the GPU must equal the oracle exactly."""
    rng = np.random.default_rng(B + T + HS)
    ints = rng.integers(-4, 5, size=(B, T, 3, NH, HS)).astype(np.float32)
    qkv = torch.from_numpy(ints)
    ref = oracle_lib.trimul_f32(ints.reshape(-1), B, T, NH * HS, NH, 0)
    out = poisoned((B, NH, T, T))
    csa.trimul_forward_f32(out, qkv.cuda(), B, T, NH * HS, NH)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    lower = ~np.triu(np.ones((T, T), dtype=bool), k=1)
    assert np.array_equal(got[..., lower], ref[..., lower])


def test_trimul_f32_lo_parts_matter(oracle_lib):
    """Inputs whose low mantissa bits carry the product: x = 1 + 2^-12 pairs, where
    one tf32 product would drop the 2^-12 terms entirely."""
    B, T, NH, HS = 1, 8, 1, 16
    x = np.full((B, T, 3, NH, HS), 1.0 + 2.0 ** -12, dtype=np.float32)
    ref = oracle_lib.trimul_f32(x.reshape(-1), B, T, NH * HS, NH, 0)
    out = poisoned((B, NH, T, T))
    csa.trimul_forward_f32(out, torch.from_numpy(x).cuda(), B, T, NH * HS, NH)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    lower = ~np.triu(np.ones((T, T), dtype=bool), k=1)
    # exact: 16 * (1 + 2^-11 + 2^-24) / 4; 3 x tf32 misses only the 2^-24 term's share.
    assert np.all(np.abs(got[..., lower] - ref[..., lower]) <= 2.0 ** -20 * ref[..., lower])
    assert np.all(got[..., lower] > 4.0 * (1.0 + 2.0 ** -12))


def test_trimul_f32_gpt2_full_size(oracle_lib):
    """The page's own configuration: (8, 1024, 3, 12, 64) fp32 uniform[-1, 1]. Mask and
    finiteness everywhere; sampled rows within the page's 1e-4 tolerance and the
    3 x tf32 bound."""
    shape = synth.TRIMUL_GPT2
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
            assert bool(torch.all(s.view(torch.int32)[upper] == NAN_BITS)), (b, h)
            assert bool(torch.all(torch.isfinite(s[~upper]))), (b, h)
    rng = np.random.default_rng(5)
    bht = np.array([(b, h, int(t)) for b in range(shape.B) for h in range(shape.NH)
                    for t in {0, T - 1, T // 2, *rng.integers(0, T, size=2).tolist()}],
                   dtype=np.int64)
    x = qkv.numpy().reshape(-1)
    ref = oracle_lib.trimul_f32_rows(x, shape.B, T, shape.C, shape.NH, bht, 0)
    ref_abs = oracle_lib.trimul_f32_rows(np.abs(x), shape.B, T, shape.C, shape.NH, bht, 0)
    idx = torch.from_numpy(bht).cuda()
    got = out[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy().astype(np.float64)
    for i, (b, h, t) in enumerate(bht):
        err = np.abs(got[i, :t + 1] - ref[i, :t + 1])
        assert float(err.max()) <= 1e-4, (b, h, t, float(err.max()))
        assert np.all(err <= F32_REL * ref_abs[i, :t + 1] + 1e-30), (b, h, t)


@pytest.mark.parametrize("B,T,NH,HS", [
    (2, 1024, 8, 128),   # Q in TMEM, one buffer, 4 chunks
    (1, 1024, 20, 96),   # Q in TMEM, one buffer, 3 chunks
    (1, 1000, 24, 64),   # Q in TMEM, two buffers, ragged T
    (1, 1024, 4, 160),   # HS > 128: Q and K chunks through the ring
])
def test_trimul_f32_many_row_blocks_per_cta(oracle_lib, B, T, NH, HS):
    """Enough tiles that every CTA walks several row blocks, so Q is reloaded (and, with
    two buffers, alternates) many times: the mask everywhere, sampled rows on both sides
    of every row-block edge within the 3 x tf32 bound, and lower-only equal bit for bit on
    and below the diagonal with nothing written above it."""
    shape, qkv = _case(B, T, NH, HS, seed=T + HS)
    out = poisoned(shape.out_shape)
    csa.trimul_forward_f32(out, qkv.cuda(), B, T, shape.C, NH)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    upper = torch.triu(torch.ones((T, T), dtype=torch.bool, device="cuda"), diagonal=1)
    bits = out.view(torch.int32)
    assert bool(torch.all(bits[..., upper] == NAN_BITS))
    assert bool(torch.all(torch.isfinite(out[..., ~upper])))
    rng = np.random.default_rng(T * HS)
    edges = sorted({0, T - 1, *range(127, T, 128), *range(128, T, 128)})
    bht = np.array([(b, h, t) for b in range(B) for h in range(NH)
                    for t in sorted(set(edges[:: max(1, len(edges) // 6)]) |
                                    set(rng.integers(0, T, size=3).tolist()))],
                   dtype=np.int64)
    x = qkv.numpy().reshape(-1)
    ref = oracle_lib.trimul_f32_rows(x, B, T, shape.C, NH, bht, 0)
    ref_abs = oracle_lib.trimul_f32_rows(np.abs(x), B, T, shape.C, NH, bht, 0)
    got = out[torch.from_numpy(bht[:, 0]).cuda(), torch.from_numpy(bht[:, 1]).cuda(),
              torch.from_numpy(bht[:, 2]).cuda()].cpu().numpy()
    _check_f32_bound(got, ref, ref_abs, f"f32 rows {(B, T, NH, HS)}")
    out2 = poisoned(shape.out_shape)
    csa.trimul_forward_f32(out2, qkv.cuda(), B, T, shape.C, NH, lower_only=True)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    bits2 = out2.view(torch.int32)
    assert bool(torch.all(bits2[..., upper] == POISON_BITS - (1 << 32)))  # as int32
    assert bool(torch.equal(bits2[..., ~upper], bits[..., ~upper]))
