"""Parity of the CUDA causal score product against the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import synth
from gpu_util import (NAN_BITS, NEG_INF_BITS, POISON_BITS, assert_close, check_trimul_full,
                      f32_bits, poisoned, trimul_case)

pytestmark = pytest.mark.gpu

# (B, T, NH, HS): tile multiples, ragged tails (T % 128 != 0, T % 4 != 0 -> plain
# stores), T smaller than a tile, several head sizes incl. HS % 16 != 0.
SHAPES = [
    (1, 64, 2, 64),     # the tiny case's shape
    (2, 1, 1, 64),
    (1, 63, 2, 64),
    (1, 65, 1, 64),
    (1, 127, 1, 64),
    (1, 128, 1, 64),
    (1, 129, 2, 64),
    (2, 200, 3, 64),
    (2, 256, 2, 64),
    (1, 300, 2, 128),
    (1, 130, 2, 128),
    (1, 100, 1, 72),
    (1, 40, 2, 8),
    (1, 97, 2, 16),
    (1, 70, 1, 256),
    (3, 384, 1, 32),
]


@pytest.mark.parametrize("B,T,NH,HS", SHAPES)
def test_trimul_parity(oracle_lib, B, T, NH, HS):
    shape, qkv = trimul_case(B, T, NH, HS, seed=B * 1000 + T * 10 + NH)
    ref = oracle_lib.trimul(synth.bf16_bits(qkv).reshape(-1), B, T, shape.C, NH, 0)
    out = poisoned(shape.out_shape)
    csa.trimul_forward(out, qkv.cuda(), B, T, shape.C, NH)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    check_trimul_full(f32_bits(out), out.cpu().numpy(), ref, NAN_BITS, f"trimul{(B, T, NH, HS)}")


def test_trimul_tiny_uniform(oracle_lib):
    """The tiny case: (1, 64, 3, 2, 64), uniform[-1, 1] seed 0, via the plain entry point."""
    shape = synth.TRIMUL_TINY
    qkv = synth.trimul_input(shape, seed=0, dist="uniform")
    ref = oracle_lib.trimul(synth.bf16_bits(qkv).reshape(-1), shape.B, shape.T, shape.C,
                            shape.NH, 0)
    out = csa.trimul(qkv.cuda())
    torch.cuda.synchronize()
    check_trimul_full(f32_bits(out), out.cpu().numpy(), ref, NAN_BITS, "tiny")


@pytest.mark.parametrize("T", [64, 129, 250])
def test_trimul_neg_inf_mask(oracle_lib, T):
    shape, qkv = trimul_case(2, T, 2, 64, seed=T)
    ref = oracle_lib.trimul(synth.bf16_bits(qkv).reshape(-1), 2, T, shape.C, 2, 1)
    out = poisoned(shape.out_shape)
    csa.trimul_forward(out, qkv.cuda(), 2, T, shape.C, 2, mask="-inf")
    torch.cuda.synchronize()
    check_trimul_full(f32_bits(out), out.cpu().numpy(), ref, NEG_INF_BITS, f"-inf T={T}")


@pytest.mark.parametrize("B,T,NH,HS", [(1, 64, 2, 64), (2, 300, 2, 64), (1, 257, 1, 128),
                                       (1, 61, 3, 64)])
def test_trimul_lower_only_leaves_upper(oracle_lib, B, T, NH, HS):
    """Lower-only mode writes t2 <= t and leaves every t2 > t element untouched."""
    shape, qkv = trimul_case(B, T, NH, HS, seed=7)
    ref = oracle_lib.trimul(synth.bf16_bits(qkv).reshape(-1), B, T, shape.C, NH, 0)
    out = poisoned(shape.out_shape)
    csa.trimul_forward(out, qkv.cuda(), B, T, shape.C, NH, lower_only=True)
    torch.cuda.synchronize()
    bits = f32_bits(out)
    upper = np.triu(np.ones((T, T), dtype=bool), k=1)
    assert np.all(bits[..., upper] == POISON_BITS)
    assert_close(out.cpu().numpy()[..., ~upper], ref[..., ~upper], "lower-only")


@pytest.mark.parametrize("B,T,NH,HS", [(1, 256, 2, 64), (2, 131, 1, 64), (1, 64, 1, 16)])
def test_trimul_integer_inputs_bit_exact(oracle_lib, B, T, NH, HS):
    """Small-integer inputs: every fp32 partial sum is exact and 1/sqrt(HS) is a power of
    two, so the GPU must equal the oracle exactly."""
    rng = np.random.default_rng(B + T)
    ints = rng.integers(-4, 5, size=(B, T, 3, NH, HS)).astype(np.float32)
    qkv = torch.from_numpy(ints).to(torch.bfloat16)
    ref = oracle_lib.trimul(synth.bf16_bits(qkv).reshape(-1), B, T, NH * HS, NH, 0)
    out = poisoned((B, NH, T, T))
    csa.trimul_forward(out, qkv.cuda(), B, T, NH * HS, NH)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    lower = ~np.triu(np.ones((T, T), dtype=bool), k=1)
    assert np.array_equal(got[..., lower], ref[..., lower])


def _full_size(oracle_lib, shape, seed, rows_per_bh=3):
    """The full-size workload in the benchmark's launch configuration: the mask and
    finiteness at every element, and sampled rows against the oracle."""
    qkv = synth.trimul_input(shape, seed=seed, dist="normal")
    out = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")
    csa.trimul_forward(out, qkv.cuda(), shape.B, shape.T, shape.C, shape.NH)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    T = shape.T
    upper = torch.triu(torch.ones((T, T), dtype=torch.bool, device="cuda"), diagonal=1)
    for b in range(shape.B):
        for h in range(shape.NH):
            s = out[b, h]
            assert bool(torch.all(s.view(torch.int32)[upper] == NAN_BITS)), (b, h)
            assert bool(torch.all(torch.isfinite(s[~upper]))), (b, h)
    rng = np.random.default_rng(seed)
    bht = []
    for b in range(shape.B):
        for h in range(shape.NH):
            ts = {0, T - 1, T // 2} | set(rng.integers(0, T, size=rows_per_bh).tolist())
            bht += [(b, h, t) for t in sorted(ts)]
    bht = np.array(bht, dtype=np.int64)
    ref = oracle_lib.trimul_rows(synth.bf16_bits(qkv).reshape(-1), shape.B, T, shape.C,
                                 shape.NH, bht, 0)
    idx = torch.from_numpy(bht).cuda()
    got = out[idx[:, 0], idx[:, 1], idx[:, 2]]
    gbits = f32_bits(got)
    gf = got.cpu().numpy()
    for i, (b, h, t) in enumerate(bht):
        assert np.all(gbits[i, t + 1:] == NAN_BITS), (b, h, t)
        assert_close(gf[i, :t + 1], ref[i, :t + 1], f"{shape} row {(b, h, t)}")


def test_trimul_gpt2_full_size(oracle_lib):
    _full_size(oracle_lib, synth.TRIMUL_GPT2, seed=0)


def test_trimul_long_context_full_size(oracle_lib):
    _full_size(oracle_lib, synth.TRIMUL_LONG, seed=0, rows_per_bh=2)


def test_trimul_many_launches_reuse_schedule_slots(oracle_lib):
    """More launches than the kernel's per-launch counter slots, alternating modes
    and streams; the last launch must still be exact (counters are reset by the
    last CTA of each launch)."""
    shape, qkv = trimul_case(2, 384, 2, 64, seed=11)
    q = qkv.cuda()
    out = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    for i in range(300):
        s = side if i % 3 == 0 else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            csa.trimul_forward(out, q, 2, 384, shape.C, 2, lower_only=(i % 2 == 1), stream=s)
        s.synchronize()
    out.view(torch.int32).fill_(-1)
    csa.trimul_forward(out, q, 2, 384, shape.C, 2)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    ref = oracle_lib.trimul(synth.bf16_bits(qkv).reshape(-1), 2, 384, shape.C, 2, 0)
    check_trimul_full(f32_bits(out), out.cpu().numpy(), ref, NAN_BITS, "after 300 launches")


def test_trimul_full_after_static_launches_in_every_slot(oracle_lib):
    """Launches with a static deal and no fill tiles (lower-only, batched NT) leave
    their counter slot untouched and skip the reset; every full-mode launch that
    follows one of them in the same slot must still store every fill tile. The
    pattern [lower-only, full, batched NT] has period 3, coprime to the 256-slot
    ring, so over 3 x 256 launches every slot serves a full launch right after a
    static one; each full launch is compared bit for bit with the first."""
    shape, qkv = trimul_case(2, 384, 2, 64, seed=12)
    q = qkv.cuda()
    ref = oracle_lib.trimul(synth.bf16_bits(qkv).reshape(-1), 2, 384, shape.C, 2, 0)
    out = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")
    out.view(torch.int32).fill_(-1)
    csa.trimul_forward(out, q, 2, 384, shape.C, 2)
    torch.cuda.synchronize()
    check_trimul_full(f32_bits(out), out.cpu().numpy(), ref, NAN_BITS, "first full launch")
    want = out.view(torch.int32).clone()
    X = torch.ones((6, 120, 64), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((6, 120, 120), dtype=torch.float32, device="cuda")
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    fulls = 0
    for i in range(3 * 256 + 3):
        kind = i % 3
        if kind == 0:
            csa.trimul_forward(out, q, 2, 384, shape.C, 2, lower_only=True)
        elif kind == 1:
            out.view(torch.int32).fill_(-1)
            csa.trimul_forward(out, q, 2, 384, shape.C, 2)
            bad += (out.view(torch.int32) != want).sum()
            fulls += 1
        else:
            csa.batch_matmul_nt(Y, X, X, 6, 120, 120, 64)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    assert fulls == 257
    assert int(bad) == 0, f"{int(bad)} words differ across the full-mode launches"
    assert torch.all(Y == 64.0)
