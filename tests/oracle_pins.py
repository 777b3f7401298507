"""Pins for the fp64 oracle: checks against something other than the oracle.

Each ``pin_*`` function takes an :class:`oracle.Oracle` and raises
AssertionError when the oracle disagrees with what the pages or the
mathematics fix. They are used twice: on the real oracle
(``test_oracle_pins.py``) and on deliberately broken copies of it
(``test_oracle_mutations.py``), where at least one pin must fail.

What each pin compares against:

* exact rational arithmetic (``fractions.Fraction``) on tiny inputs, a method
  that does no floating-point rounding at all;
* a library routine: ``torch.matmul`` in float64, whose lower triangle scaled
  by 1/sqrt(HS) is the causal score ("llm.c dev/cuda/trimat_forward.cu",
  the referee computes q.k only for t2 <= t), and X @ W.T for the dense layer
  ("DietCode ... test_local_padding", Y[i, j] += X[i, k] * W[j, k]);
* closed forms (all-ones, one-hot, small integers whose sums are exact);
* invariants: mask positions and counts, causality under perturbation, head
  permutation, zero padding along the reduction axis (local padding), row
  independence, transposition.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import torch

from causal_attention_score_gb300 import synth

MASK_NAN = 0
MASK_NEG_INF = 1


# ---------------------------------------------------------------- helpers --

def _u16_to_f32(u: np.ndarray) -> np.ndarray:
    return (u.astype(np.uint32) << 16).view(np.float32)


def _bits_of(values: np.ndarray) -> np.ndarray:
    """bf16 patterns of float values that are exactly representable in bf16."""
    f = np.asarray(values, dtype=np.float32)
    bits = f.view(np.uint32)
    if np.any(bits & 0xFFFF):
        raise ValueError("value not exactly representable in bf16")
    return (bits >> 16).astype(np.uint16)


def _qkv_from_parts(Q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Pack float arrays Q, K, V of shape (B, T, NH, HS) into (B, T, 3, NH, HS) bf16 bits."""
    qkv = np.stack([Q, K, V], axis=2)
    return _bits_of(qkv)


def _random_qkv(B, T, NH, HS, seed, dist="uniform"):
    shape = synth.TrimulShape(B=B, T=T, C=NH * HS, NH=NH)
    t = synth.trimul_input(shape, seed=seed, dist=dist)
    return synth.bf16_bits(t).reshape(-1)


def _random_qkv_f32(B, T, NH, HS, seed, dist="uniform"):
    shape = synth.TrimulShape(B=B, T=T, C=NH * HS, NH=NH)
    return synth.trimul_input_f32(shape, seed=seed, dist=dist).numpy().reshape(-1)


def _split_qk(qkv_u16, B, T, NH, HS):
    f = _u16_to_f32(qkv_u16).astype(np.float64).reshape(B, T, 3, NH, HS)
    Q = f[:, :, 0].transpose(0, 2, 1, 3)  # (B, NH, T, HS)
    K = f[:, :, 1].transpose(0, 2, 1, 3)
    return Q, K


# ------------------------------------------------------- score product pins --

def pin_trimul_exact_rational(o):
    """Brute force in exact rationals on tiny inputs, then one division by sqrt(HS)."""
    for (B, T, NH, HS, seed) in [(2, 7, 2, 8, 3), (1, 5, 1, 16, 4), (1, 1, 3, 8, 5)]:
        C = NH * HS
        qkv = _random_qkv(B, T, NH, HS, seed)
        f = _u16_to_f32(qkv).reshape(B, T, 3, NH, HS)
        out = o.trimul(qkv, B, T, C, NH, MASK_NAN)
        root = math.sqrt(HS)
        for b in range(B):
            for h in range(NH):
                for t in range(T):
                    for t2 in range(T):
                        got = out[b, h, t, t2]
                        if t2 > t:
                            assert math.isnan(got), (b, h, t, t2, got)
                            continue
                        exact = sum((Fraction(float(f[b, t, 0, h, d])) * Fraction(float(f[b, t2, 1, h, d]))
                                     for d in range(HS)), Fraction(0))
                        want = float(exact) / root
                        assert abs(got - want) <= 1e-14 * (1.0 + abs(want)), (b, h, t, t2, got, want)


def pin_trimul_matmul_identity(o):
    """The unmasked triangle equals the lower half of a full Q K^T (torch fp64) / sqrt(HS)."""
    for (B, T, NH, HS, seed, dist) in [(2, 37, 3, 24, 11, "normal"), (1, 130, 2, 64, 12, "uniform")]:
        C = NH * HS
        qkv = _random_qkv(B, T, NH, HS, seed, dist)
        Q, K = _split_qk(qkv, B, T, NH, HS)
        full = torch.matmul(torch.from_numpy(Q), torch.from_numpy(K).transpose(-1, -2)).numpy()
        want = full / math.sqrt(HS)
        out = o.trimul(qkv, B, T, C, NH, MASK_NAN)
        lower = np.tril(np.ones((T, T), dtype=bool))
        got_l = out[..., lower]
        want_l = want[..., lower]
        assert np.all(np.isfinite(got_l))
        assert np.max(np.abs(got_l - want_l) / (1.0 + np.abs(want_l))) <= 1e-12
        assert np.all(np.isnan(out[..., ~lower]))


def pin_trimul_closed_forms(o):
    """All-ones rows give sqrt(HS); one-hot rows give delta / sqrt(HS)."""
    for HS in (4, 16, 64, 128, 256):
        B, T, NH = 1, 6, 2
        ones = np.ones((B, T, NH, HS), dtype=np.float32)
        qkv = _qkv_from_parts(ones, ones, ones * 2)
        out = o.trimul(qkv, B, T, NH * HS, NH, MASK_NAN)
        lower = np.tril(np.ones((T, T), dtype=bool))
        # HS / sqrt(HS) == sqrt(HS): exact for perfect squares, within one ulp otherwise.
        want = math.sqrt(HS)
        err = np.abs(out[..., lower] - want)
        if math.isqrt(HS) ** 2 == HS:
            assert np.all(err == 0.0), (HS, out[..., lower][:4])
        else:
            assert np.all(err <= 2 * np.spacing(want)), HS
    # one-hot: Q[t] = e_{t mod HS}, K[t2] = e_{(t2 + 1) mod HS}
    B, T, NH, HS = 1, 9, 1, 4
    Q = np.zeros((B, T, NH, HS), np.float32)
    K = np.zeros((B, T, NH, HS), np.float32)
    for t in range(T):
        Q[0, t, 0, t % HS] = 1.0
        K[0, t, 0, (t + 1) % HS] = 1.0
    out = o.trimul(_qkv_from_parts(Q, K, np.zeros_like(Q)), B, T, NH * HS, NH, MASK_NAN)
    for t in range(T):
        for t2 in range(t + 1):
            want = 0.5 if (t % HS) == ((t2 + 1) % HS) else 0.0  # 1/sqrt(4)
            assert out[0, 0, t, t2] == want, (t, t2, out[0, 0, t, t2])


def pin_trimul_integer_exact(o):
    """Small-integer inputs: every sum is exact; compare with int64 arithmetic."""
    rng = np.random.default_rng(7)
    for (B, T, NH, HS) in [(2, 11, 2, 64), (1, 8, 3, 16), (1, 5, 1, 4)]:
        ints = rng.integers(-4, 5, size=(B, T, 3, NH, HS)).astype(np.int64)
        qkv = _bits_of(ints.astype(np.float32))
        out = o.trimul(qkv, B, T, NH * HS, NH, MASK_NAN)
        Qi = ints[:, :, 0].transpose(0, 2, 1, 3)
        Ki = ints[:, :, 1].transpose(0, 2, 1, 3)
        dots = np.einsum("bhtd,bhsd->bhts", Qi, Ki)  # exact int64
        root = math.isqrt(HS)  # 8, 4, 2: exact divisions
        for t in range(T):
            for t2 in range(t + 1):
                assert np.array_equal(out[:, :, t, t2], dots[:, :, t, t2] / root)


def pin_trimul_index_roles(o):
    """Query rows index t, key rows index t2, keys sit C after the queries, V is ignored,
    heads and batches are kept apart. Built so that any swap changes the value."""
    B, T, NH, HS = 2, 6, 3, 16
    Q = np.zeros((B, T, NH, HS), np.float32)
    K = np.zeros((B, T, NH, HS), np.float32)
    V = np.full((B, T, NH, HS), 96.0, np.float32)
    for b in range(B):
        for t in range(T):
            for h in range(NH):
                Q[b, t, h, 0] = t + 1
                Q[b, t, h, 1] = h + 1
                K[b, t, h, 0] = 1.0
                K[b, t, h, 1] = (b + 1) * (t + 1)
    out = o.trimul(_qkv_from_parts(Q, K, V), B, T, NH * HS, NH, MASK_NAN)
    for b in range(B):
        for h in range(NH):
            for t in range(T):
                for t2 in range(t + 1):
                    want = ((t + 1) + (h + 1) * (b + 1) * (t2 + 1)) / 4.0
                    assert out[b, h, t, t2] == want, (b, h, t, t2, out[b, h, t, t2], want)


def pin_trimul_mask_and_causality(o):
    """Mask count T(T-1)/2 per head at exactly t2 > t; -inf mode; causality under perturbation."""
    B, T, NH, HS = 2, 19, 2, 8
    C = NH * HS
    qkv = _random_qkv(B, T, NH, HS, 21)
    out = o.trimul(qkv, B, T, C, NH, MASK_NAN)
    upper = np.triu(np.ones((T, T), dtype=bool), k=1)
    nan = np.isnan(out)
    assert nan.sum() == B * NH * T * (T - 1) // 2
    assert np.array_equal(nan, np.broadcast_to(upper, out.shape))
    out_inf = o.trimul(qkv, B, T, C, NH, MASK_NEG_INF)
    assert np.all(out_inf[..., upper] == -np.inf)
    assert np.array_equal(out_inf[..., ~upper], out[..., ~upper])
    # changing key row s touches only column s at rows t >= s
    s = 7
    pert = qkv.reshape(B, T, 3, NH, HS).copy()
    pert[:, s, 1] = _bits_of(np.full((B, NH, HS), 0.75, np.float32))
    out_p = o.trimul(pert.reshape(-1), B, T, C, NH, MASK_NAN)
    changed = ~((out_p == out) | (np.isnan(out_p) & np.isnan(out)))
    allowed = np.zeros((T, T), dtype=bool)
    allowed[s:, s] = True
    assert not np.any(changed & ~allowed)
    assert np.any(changed[..., s:, s])
    # permuting the heads of the input permutes the heads of the output
    perm = [1, 0]
    permuted = qkv.reshape(B, T, 3, NH, HS)[:, :, :, perm].copy().reshape(-1)
    out_h = o.trimul(permuted, B, T, C, NH, MASK_NAN)
    assert np.array_equal(np.nan_to_num(out_h), np.nan_to_num(out[:, perm]))


def pin_trimul_rows(o):
    """Sampled rows agree with the full tensor."""
    B, T, NH, HS = 2, 23, 3, 8
    qkv = _random_qkv(B, T, NH, HS, 31)
    full = o.trimul(qkv, B, T, NH * HS, NH, MASK_NAN)
    bht = np.array([[0, 0, 0], [1, 2, 22], [0, 1, 11], [1, 0, 5]])
    rows = o.trimul_rows(qkv, B, T, NH * HS, NH, bht, MASK_NAN)
    for i, (b, h, t) in enumerate(bht):
        assert np.array_equal(np.nan_to_num(rows[i], nan=7.0), np.nan_to_num(full[b, h, t], nan=7.0))


# ------------------------------------------------------------ dense pins --

def _dense_random(M, I, H, seed):
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=seed)
    return synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1)


def pin_dense_exact_rational(o):
    M, I, H = 3, 5, 4
    x, w = _dense_random(M, I, H, 41)
    xf, wf = _u16_to_f32(x).reshape(M, I), _u16_to_f32(w).reshape(H, I)
    Y = o.dense(x, w, M, I, H)
    for i in range(M):
        for j in range(H):
            exact = sum((Fraction(float(xf[i, k])) * Fraction(float(wf[j, k])) for k in range(I)),
                        Fraction(0))
            assert abs(Y[i, j] - float(exact)) <= 1e-15 * (1 + abs(float(exact)))


def pin_dense_matmul_identity(o):
    for (M, I, H, seed) in [(37, 45, 29, 42), (130, 770, 70, 43)]:
        x, w = _dense_random(M, I, H, seed)
        xf = torch.from_numpy(_u16_to_f32(x).astype(np.float64).reshape(M, I))
        wf = torch.from_numpy(_u16_to_f32(w).astype(np.float64).reshape(H, I))
        want = (xf @ wf.T).numpy()
        Y = o.dense(x, w, M, I, H)
        assert np.max(np.abs(Y - want) / (1 + np.abs(want))) <= 1e-12


def pin_dense_integer_exact(o):
    rng = np.random.default_rng(9)
    M, I, H = 17, 770, 13
    Xi = rng.integers(-4, 5, size=(M, I)).astype(np.int64)
    Wi = rng.integers(-4, 5, size=(H, I)).astype(np.int64)
    Y = o.dense(_bits_of(Xi.astype(np.float32)), _bits_of(Wi.astype(np.float32)), M, I, H)
    assert np.array_equal(Y, (Xi @ Wi.T).astype(np.float64))


def pin_dense_local_padding(o):
    """Zero columns appended along I change nothing; rows are independent;
    swapping X and W transposes Y."""
    M, I, H = 9, 13, 6
    x, w = _dense_random(M, I, H, 44)
    Y = o.dense(x, w, M, I, H)
    pad = 19
    xp = np.concatenate([x.reshape(M, I), np.zeros((M, pad), np.uint16)], axis=1)
    wp = np.concatenate([w.reshape(H, I), np.zeros((H, pad), np.uint16)], axis=1)
    assert np.array_equal(o.dense(xp.reshape(-1), wp.reshape(-1), M, I + pad, H), Y)
    one = o.dense(x.reshape(M, I)[4:5].reshape(-1), w, 1, I, H)
    assert np.array_equal(one[0], Y[4])
    rows = o.dense_rows(x, w, M, I, H, np.array([8, 0, 4]))
    assert np.array_equal(rows, Y[[8, 0, 4]])
    Yt = o.dense(w, x, H, I, M)
    assert np.array_equal(Yt, Y.T)


# ------------------------------------------------------ batched NT pins --

def _bmm_random(batch, T1, T2, D, seed):
    X, W = synth.bmm_input(synth.BmmShape(batch=batch, T1=T1, T2=T2, D=D), seed=seed)
    return synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1)


def pin_bmm_exact_rational(o):
    batch, T1, T2, D = 2, 3, 4, 5
    x, w = _bmm_random(batch, T1, T2, D, 51)
    xf = _u16_to_f32(x).reshape(batch, T1, D)
    wf = _u16_to_f32(w).reshape(batch, T2, D)
    Y = o.bmm_nt(x, w, batch, T1, T2, D)
    for i in range(batch):
        for j in range(T1):
            for k in range(T2):
                exact = sum((Fraction(float(xf[i, j, l])) * Fraction(float(wf[i, k, l]))
                             for l in range(D)), Fraction(0))
                assert abs(Y[i, j, k] - float(exact)) <= 1e-15 * (1 + abs(float(exact)))


def pin_bmm_matmul_identity(o):
    for (batch, T1, T2, D, seed) in [(3, 17, 29, 24, 52), (2, 120, 120, 64, 53)]:
        x, w = _bmm_random(batch, T1, T2, D, seed)
        xf = torch.from_numpy(_u16_to_f32(x).astype(np.float64).reshape(batch, T1, D))
        wf = torch.from_numpy(_u16_to_f32(w).astype(np.float64).reshape(batch, T2, D))
        want = torch.bmm(xf, wf.transpose(1, 2)).numpy()
        Y = o.bmm_nt(x, w, batch, T1, T2, D)
        assert np.max(np.abs(Y - want) / (1 + np.abs(want))) <= 1e-12


def pin_bmm_integer_exact_and_structure(o):
    """Small integers: exact against int64; swapping X and W transposes each
    batch; each batch depends only on its own inputs."""
    rng = np.random.default_rng(13)
    batch, T1, T2, D = 3, 9, 7, 16
    Xi = rng.integers(-4, 5, size=(batch, T1, D)).astype(np.int64)
    Wi = rng.integers(-4, 5, size=(batch, T2, D)).astype(np.int64)
    xb, wb = _bits_of(Xi.astype(np.float32)), _bits_of(Wi.astype(np.float32))
    Y = o.bmm_nt(xb, wb, batch, T1, T2, D)
    assert np.array_equal(Y, np.einsum("bjl,bkl->bjk", Xi, Wi).astype(np.float64))
    Yt = o.bmm_nt(wb, xb, batch, T2, T1, D)
    assert np.array_equal(Yt, Y.transpose(0, 2, 1))
    Wi2 = Wi.copy()
    Wi2[1] = -Wi2[1]
    Y2 = o.bmm_nt(xb, _bits_of(Wi2.astype(np.float32)), batch, T1, T2, D)
    assert np.array_equal(Y2[[0, 2]], Y[[0, 2]]) and np.array_equal(Y2[1], -Y[1])


def pin_bmm_vs_causal_score(o):
    """The causal score of "trimat_forward.cu" is the lower triangle of the batched
    NT product of its Q and K heads, divided by sqrt(HS); checked between two
    independently written oracle functions."""
    B, T, NH, HS = 2, 21, 2, 16
    qkv = _random_qkv(B, T, NH, HS, 61)
    q5 = qkv.reshape(B, T, 3, NH, HS)
    Q = np.ascontiguousarray(q5[:, :, 0].transpose(0, 2, 1, 3)).reshape(-1)
    K = np.ascontiguousarray(q5[:, :, 1].transpose(0, 2, 1, 3)).reshape(-1)
    Y = o.bmm_nt(Q, K, B * NH, T, T, HS).reshape(B, NH, T, T)
    S = o.trimul(qkv, B, T, NH * HS, NH, MASK_NAN)
    lower = np.tril(np.ones((T, T), dtype=bool))
    assert np.array_equal(S[..., lower], Y[..., lower] / math.sqrt(HS))


# -------------------------------------------------------- softmax pins --

def pin_softmax_matches_library_softmax(o):
    """Each row equals scipy.special.softmax of the causal score row (t2 <= t); 0 above."""
    import scipy.special
    for (B, T, NH, HS, seed, dist) in [(2, 37, 3, 24, 71, "normal"), (1, 130, 2, 64, 72, "uniform")]:
        qkv = _random_qkv(B, T, NH, HS, seed, dist)
        P = o.causal_softmax(qkv, B, T, NH * HS, NH)
        S = o.trimul(qkv, B, T, NH * HS, NH, MASK_NAN)
        for b in range(B):
            for h in range(NH):
                for t in range(T):
                    want = scipy.special.softmax(S[b, h, t, :t + 1])
                    assert np.max(np.abs(P[b, h, t, :t + 1] - want)) <= 1e-14
                    assert np.all(P[b, h, t, t + 1:] == 0.0)
        assert np.max(np.abs(P.sum(axis=-1) - 1.0)) <= 1e-12


def pin_softmax_large_scores_and_closed_form(o):
    """Scores beyond 709 (where exp overflows in fp64) stay finite and exact against
    scipy (the row maximum is subtracted); equal scores give 1/(t+1)."""
    import scipy.special
    B, T, NH, HS = 1, 12, 1, 16
    Q = np.zeros((B, T, NH, HS), np.float32)
    K = np.zeros((B, T, NH, HS), np.float32)
    for t in range(T):
        Q[0, t, 0, 0] = 64.0 * (1 if t % 2 else -1)
        K[0, t, 0, 0] = float(t % 5 - 2) * 16.0  # q.k/4 in [-512, 512]
        Q[0, t, 0, 1] = 32.0
        K[0, t, 0, 1] = float(t) * 8.0             # + up to 704: exp() of it overflows fp64
    qkv = _qkv_from_parts(Q, K, np.zeros_like(Q))
    P = o.causal_softmax(qkv, B, T, NH * HS, NH)
    S = o.trimul(qkv, B, T, NH * HS, NH, MASK_NAN)
    assert np.nanmax(S) > 720
    assert np.all(np.isfinite(P))
    for t in range(T):
        assert np.max(np.abs(P[0, 0, t, :t + 1] - scipy.special.softmax(S[0, 0, t, :t + 1]))) <= 1e-14
    ones = np.ones((1, 9, 1, 8), np.float32)
    P1 = o.causal_softmax(_qkv_from_parts(ones, ones, ones), 1, 9, 8, 1)
    for t in range(9):
        assert np.all(P1[0, 0, t, :t + 1] == 1.0 / (t + 1))
        assert np.all(P1[0, 0, t, t + 1:] == 0.0)


def pin_softmax_causality_and_rows(o):
    """Changing key row s changes exactly the rows t >= s; sampled rows match."""
    B, T, NH, HS = 1, 17, 2, 8
    qkv = _random_qkv(B, T, NH, HS, 73)
    P = o.causal_softmax(qkv, B, T, NH * HS, NH)
    s = 6
    pert = qkv.reshape(B, T, 3, NH, HS).copy()
    pert[:, s, 1] = _bits_of(np.full((B, NH, HS), 0.5, np.float32))
    P2 = o.causal_softmax(pert.reshape(-1), B, T, NH * HS, NH)
    changed_rows = np.any(P2 != P, axis=-1)  # (B, NH, T)
    assert not np.any(changed_rows[..., :s]) and np.all(changed_rows[..., s:])
    bht = np.array([[0, 0, 0], [0, 1, 16], [0, 1, 5]])
    rows = o.causal_softmax_rows(qkv, B, T, NH * HS, NH, bht)
    for i, (b, h, t) in enumerate(bht):
        assert np.array_equal(rows[i], P[b, h, t])


# ------------------------------------------ score product, fp32 inputs pins --

def pin_trimul_f32_exact_rational(o):
    """fp32 inputs finer than bf16, through exact rationals, then one division by sqrt(HS)."""
    for (B, T, NH, HS, seed) in [(2, 6, 2, 8, 11), (1, 4, 1, 12, 12)]:
        C = NH * HS
        x = _random_qkv_f32(B, T, NH, HS, seed)
        assert np.any(x.view(np.uint32) & 0xFFFF), "inputs must not all be bf16 values"
        f = x.reshape(B, T, 3, NH, HS)
        out = o.trimul_f32(x, B, T, C, NH, MASK_NAN)
        root = math.sqrt(HS)
        for b in range(B):
            for h in range(NH):
                for t in range(T):
                    for t2 in range(T):
                        if t2 > t:
                            assert math.isnan(out[b, h, t, t2])
                            continue
                        exact = sum(Fraction(float(f[b, t, 0, h, d])) * Fraction(float(f[b, t2, 1, h, d]))
                                    for d in range(HS))
                        want = float(exact) / root
                        assert abs(out[b, h, t, t2] - want) <= 1e-15 * (1.0 + abs(want))


def pin_trimul_f32_matmul_identity(o):
    """Lower triangle of torch.matmul(Q, K^T) in float64 over the fp32 inputs, over
    sqrt(HS); -inf above (mask kind 1)."""
    B, T, NH, HS = 2, 33, 3, 20
    x = _random_qkv_f32(B, T, NH, HS, 13, "normal")
    out = torch.from_numpy(o.trimul_f32(x, B, T, NH * HS, NH, MASK_NEG_INF))
    f = torch.from_numpy(x.reshape(B, T, 3, NH, HS).astype(np.float64))
    Q = f[:, :, 0].permute(0, 2, 1, 3)
    K = f[:, :, 1].permute(0, 2, 1, 3)
    ref = torch.matmul(Q, K.transpose(-1, -2)) / math.sqrt(HS)
    lower = torch.tril(torch.ones(T, T, dtype=torch.bool))
    assert torch.allclose(out[..., lower], ref[..., lower], rtol=1e-13, atol=1e-13)
    assert torch.all(torch.isneginf(out[..., ~lower]))


def pin_trimul_f32_agrees_with_bf16_referee(o):
    """On inputs that are bf16 values, the fp32-input and bf16-input referees are the
    same function, to the bit (both widen exactly and sum in the same order)."""
    B, T, NH, HS = 2, 40, 2, 16
    u16 = _random_qkv(B, T, NH, HS, 14)
    a = o.trimul_f32(_u16_to_f32(u16), B, T, NH * HS, NH, MASK_NAN)
    b = o.trimul(u16, B, T, NH * HS, NH, MASK_NAN)
    assert np.array_equal(a, b, equal_nan=True)


def pin_trimul_f32_causality_and_rows(o):
    """Changing key row s changes exactly column s of rows t >= s; changing query row t
    changes exactly row t's columns t2 <= t; sampled rows match."""
    B, T, NH, HS = 2, 9, 2, 8
    x = _random_qkv_f32(B, T, NH, HS, 15)
    P = o.trimul_f32(x, B, T, NH * HS, NH, MASK_NAN)
    f = x.reshape(B, T, 3, NH, HS)
    s = 4
    k2 = f.copy()
    k2[1, s, 1, 0] += 0.375
    P2 = o.trimul_f32(k2.reshape(-1), B, T, NH * HS, NH, MASK_NAN)
    diff = ~((P2 == P) | (np.isnan(P2) & np.isnan(P)))
    want = np.zeros_like(diff)
    want[1, 0, s:, s] = True
    assert np.array_equal(diff, want)
    q2 = f.copy()
    q2[0, s, 0, 1] -= 0.25
    P3 = o.trimul_f32(q2.reshape(-1), B, T, NH * HS, NH, MASK_NAN)
    diff = ~((P3 == P) | (np.isnan(P3) & np.isnan(P)))
    want = np.zeros_like(diff)
    want[0, 1, s, :s + 1] = True
    assert np.array_equal(diff, want)
    bht = np.array([[0, 0, 0], [1, 1, 8], [0, 1, 4]])
    rows = o.trimul_f32_rows(x, B, T, NH * HS, NH, bht, MASK_NAN)
    for i, (b, h, t) in enumerate(bht):
        assert np.array_equal(rows[i], P[b, h, t], equal_nan=True)


SOFTMAX_PINS = [pin_softmax_matches_library_softmax, pin_softmax_large_scores_and_closed_form,
                pin_softmax_causality_and_rows]

BMM_PINS = [pin_bmm_exact_rational, pin_bmm_matmul_identity, pin_bmm_integer_exact_and_structure,
            pin_bmm_vs_causal_score]

TRIMUL_PINS = [pin_trimul_exact_rational, pin_trimul_matmul_identity, pin_trimul_closed_forms,
               pin_trimul_integer_exact, pin_trimul_index_roles, pin_trimul_mask_and_causality,
               pin_trimul_rows]
DENSE_PINS = [pin_dense_exact_rational, pin_dense_matmul_identity, pin_dense_integer_exact,
              pin_dense_local_padding]
TRIMUL_F32_PINS = [pin_trimul_f32_exact_rational, pin_trimul_f32_matmul_identity,
                   pin_trimul_f32_agrees_with_bf16_referee, pin_trimul_f32_causality_and_rows]

ALL_PINS = TRIMUL_PINS + DENSE_PINS + BMM_PINS + SOFTMAX_PINS + TRIMUL_F32_PINS
