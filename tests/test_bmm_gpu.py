"""Parity of the CUDA batched NT product (DietCode's BatchMatmulNT) against the
fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import synth
from gpu_util import assert_close, poisoned

pytestmark = pytest.mark.gpu

# (batch, T1, T2, D): the page's B*NH=192, T=120, D=64 case; T1 != T2; T2 % 4 != 0
# (plain stores); tails past 128; D % 16 != 0; small and large D.
SHAPES = [
    (192, 120, 120, 64),
    (3, 1, 1, 64),
    (2, 130, 77, 64),
    (4, 256, 384, 128),
    (1, 300, 300, 72),
    (2, 64, 200, 8),
    (5, 129, 131, 256),
    (7, 33, 257, 16),
]


def _run(X, W, batch, T1, T2, D):
    Y = poisoned((batch, T1, T2))
    csa.batch_matmul_nt(Y, X.cuda(), W.cuda(), batch, T1, T2, D)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    return Y


@pytest.mark.parametrize("batch,T1,T2,D", SHAPES)
def test_bmm_nt_parity(oracle_lib, batch, T1, T2, D):
    X, W = synth.bmm_input(synth.BmmShape(batch, T1, T2, D), seed=batch + T1 + T2 + D)
    ref = oracle_lib.bmm_nt(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                            batch, T1, T2, D)
    Y = _run(X, W, batch, T1, T2, D)
    assert_close(Y.cpu().numpy(), ref, f"bmm_nt{(batch, T1, T2, D)}")


@pytest.mark.parametrize("batch,T1,T2,D", [(3, 120, 120, 64), (2, 200, 131, 32)])
def test_bmm_nt_integer_inputs_bit_exact(oracle_lib, batch, T1, T2, D):
    rng = np.random.default_rng(batch * T1)
    X = torch.from_numpy(rng.integers(-4, 5, size=(batch, T1, D)).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy(rng.integers(-4, 5, size=(batch, T2, D)).astype(np.float32)).to(torch.bfloat16)
    ref = oracle_lib.bmm_nt(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                            batch, T1, T2, D)
    Y = _run(X, W, batch, T1, T2, D)
    assert np.array_equal(Y.cpu().numpy().astype(np.float64), ref)


def test_bmm_nt_matches_unmasked_scores_of_packed_qkv():
    """On the same heads, the batched NT product over sqrt(HS) equals trimul's lower
    triangle (both run on the GPU; one through the packed layout, one through
    separate tensors)."""
    B, T, NH, HS = 2, 200, 3, 64
    qkv = synth.trimul_input(synth.TrimulShape(B=B, T=T, C=NH * HS, NH=NH), seed=4).cuda()
    Q = qkv[:, :, 0].permute(0, 2, 1, 3).contiguous().reshape(B * NH, T, HS)
    K = qkv[:, :, 1].permute(0, 2, 1, 3).contiguous().reshape(B * NH, T, HS)
    Y = torch.empty((B * NH, T, T), dtype=torch.float32, device="cuda")
    csa.batch_matmul_nt(Y, Q, K, B * NH, T, T, HS)
    S = csa.trimul(qkv)
    torch.cuda.synchronize()
    lower = torch.tril(torch.ones((T, T), dtype=torch.bool, device="cuda"))
    got = S.reshape(B * NH, T, T)[:, lower]
    want = Y[:, lower] * (1.0 / 8.0)
    assert torch.equal(got, want)
