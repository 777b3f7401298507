"""The largest and most numerous cases each entry point takes in one launch (GPU):
very long sequences (row blocks of 128 tiles, the longest work-list decodes), thousands
of one-tile heads or batches, and a tall ragged dense layer, checked on sampled rows
against the fp64 oracle and on every element for the mask / zero / normalisation
properties."""
import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import synth
from gpu_util import (NAN_BITS, POISON_BITS, assert_close, assert_softmax_close, f32_bits,
                      poisoned, softmax_abs_scores, softmax_rel_bound)

pytestmark = pytest.mark.gpu


def _edge_rows(T, rng, extra=4):
    """Rows on both sides of every few row-block edges, the first and last, and a few more."""
    edges = sorted({0, T - 1} | {e for k in range(128, T, 128 * max(1, T // 1024))
                                 for e in (k - 1, k)})
    return sorted(set(edges) | set(rng.integers(0, T, size=extra).tolist()))


def _upper_is(out_bh: torch.Tensor, bits: int) -> bool:
    """Every element above the diagonal of one (T, T) plane has the given bit pattern,
    checked one 1024-row band at a time (no T x T index tensor)."""
    T = out_bh.shape[-1]
    v = out_bh.view(torch.int32)
    want = bits - (1 << 32) if bits >= 1 << 31 else bits
    cols = torch.arange(T, device=out_bh.device)
    for r0 in range(0, T, 1024):
        rows = torch.arange(r0, min(T, r0 + 1024), device=out_bh.device)
        band = v[r0:r0 + len(rows)]
        upper = cols[None, :] > rows[:, None]
        if not bool(torch.all(band[upper] == want)):
            return False
    return True


def test_trimul_sequence_16384_full_and_lower_only(oracle_lib):
    shape = synth.TrimulShape(B=1, T=16384, C=64, NH=1)
    qkv = synth.trimul_input(shape, seed=7)
    out = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")
    csa.trimul_forward(out, qkv.cuda(), 1, shape.T, shape.C, 1)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    T = shape.T
    assert _upper_is(out[0, 0], NAN_BITS)
    rows = _edge_rows(T, np.random.default_rng(1))
    bht = np.array([(0, 0, t) for t in rows], dtype=np.int64)
    ref = oracle_lib.trimul_rows(synth.bf16_bits(qkv).reshape(-1), 1, T, shape.C, 1, bht, 0)
    got = out[0, 0, torch.tensor(rows, device="cuda")].cpu().numpy()
    for i, t in enumerate(rows):
        assert_close(got[i, :t + 1], ref[i, :t + 1], f"T=16384 row {t}")
    lower = poisoned(shape.out_shape)
    csa.trimul_forward(lower, qkv.cuda(), 1, T, shape.C, 1, lower_only=True)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    assert _upper_is(lower[0, 0], POISON_BITS)
    assert bool(torch.equal(torch.tril(lower[0, 0]), torch.tril(out[0, 0])))


def test_softmax_sequence_16384(oracle_lib):
    shape = synth.TrimulShape(B=1, T=16384, C=128, NH=1)
    qkv = synth.trimul_input(shape, seed=8)
    att = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")
    csa.causal_softmax_forward(att, qkv.cuda(), 1, shape.T, shape.C, 1)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    T = shape.T
    assert _upper_is(att[0, 0], 0)
    sums = att[0, 0].sum(dim=-1, dtype=torch.float64)
    assert float((sums - 1).abs().max()) <= 1e-4
    rows = _edge_rows(T, np.random.default_rng(2))
    bht = np.array([(0, 0, t) for t in rows], dtype=np.int64)
    ref = oracle_lib.causal_softmax_rows(synth.bf16_bits(qkv).reshape(-1), 1, T, shape.C, 1, bht)
    got = att[0, 0, torch.tensor(rows, device="cuda")].cpu().numpy()
    assert_close(got, ref, "softmax T=16384 rows")
    rel = softmax_rel_bound(softmax_abs_scores(oracle_lib, qkv, 1, T, shape.C, 1, bht),
                            bht[:, 2], shape.HS)
    rel = np.where(np.arange(T)[None, :] > bht[:, 2:3], np.inf, rel)
    assert_softmax_close(got, ref, rel, "softmax T=16384 rows (relative bound)")


def test_4096_one_tile_heads(oracle_lib):
    """B = 64, NH = 64, T = 64: 4096 (b, h) problems of one (diagonal) tile each, scores
    and softmax, every element against the oracle."""
    shape = synth.TrimulShape(B=64, T=64, C=64 * 64, NH=64)
    qkv = synth.trimul_input(shape, seed=9)
    bits = synth.bf16_bits(qkv).reshape(-1)
    out = poisoned(shape.out_shape)
    csa.trimul_forward(out, qkv.cuda(), 64, 64, shape.C, 64)
    att = poisoned(shape.out_shape)
    csa.causal_softmax_forward(att, qkv.cuda(), 64, 64, shape.C, 64)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    ref = oracle_lib.trimul(bits, 64, 64, shape.C, 64, 0)
    ob = f32_bits(out)
    upper = np.triu(np.ones((64, 64), dtype=bool), k=1)
    assert np.all(ob[..., upper] == NAN_BITS)
    assert_close(out.cpu().numpy()[..., ~upper], ref[..., ~upper], "4096 heads scores")
    sref = oracle_lib.causal_softmax(bits, 64, 64, shape.C, 64)
    assert_close(att.cpu().numpy(), sref, "4096 heads softmax")


def test_bmm_nt_20000_tiny_batches(oracle_lib):
    batch, T1, T2, D = 20000, 8, 5, 16
    X, W = synth.bmm_input(synth.BmmShape(batch=batch, T1=T1, T2=T2, D=D), seed=3)
    Y = poisoned((batch, T1, T2))
    csa.batch_matmul_nt(Y, X.cuda(), W.cuda(), batch, T1, T2, D)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    ref = oracle_lib.bmm_nt(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                            batch, T1, T2, D)
    assert_close(Y.cpu().numpy(), ref, "20000 batches")


def test_dense_65536_ragged_rows(oracle_lib):
    """A tall ragged layer (1540-byte rows, realigned copy + TMA), sampled rows."""
    M, I, H = 65536, 770, 96
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=4)
    Y = poisoned((M, H))
    csa.dense_xwt(Y, X.cuda(), W.cuda(), M, I, H)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    assert bool(torch.all(torch.isfinite(Y)))
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], np.random.default_rng(4).integers(0, M, 40)]))
    ref = oracle_lib.dense_rows(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                                M, I, H, rows)
    assert_close(Y[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, "dense 65536 rows")


def test_trimul_f32_sequence_8192(oracle_lib):
    shape = synth.TrimulShape(B=1, T=8192, C=128, NH=1)
    qkv = synth.trimul_input_f32(shape, seed=10)
    out = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")
    csa.trimul_forward_f32(out, qkv.cuda(), 1, shape.T, shape.C, 1)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    T = shape.T
    assert _upper_is(out[0, 0], NAN_BITS)
    rows = _edge_rows(T, np.random.default_rng(3))
    bht = np.array([(0, 0, t) for t in rows], dtype=np.int64)
    x = qkv.numpy().reshape(-1)
    ref = oracle_lib.trimul_f32_rows(x, 1, T, shape.C, 1, bht, 0)
    ref_abs = oracle_lib.trimul_f32_rows(np.abs(x), 1, T, shape.C, 1, bht, 0)
    got = out[0, 0, torch.tensor(rows, device="cuda")].cpu().numpy().astype(np.float64)
    lower = ~np.isnan(ref)
    err = np.abs(got[lower] - ref[lower])
    assert float((err / (2.0 ** -15 * ref_abs[lower] + 1e-30)).max()) <= 1.0
