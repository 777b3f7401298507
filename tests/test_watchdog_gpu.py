"""The device watchdog: a withheld tile load makes a bounded wait run out; the
kernel reports CSA_ERR_TIMEOUT through the status word and returns, and the
context stays usable (no fault, no hang)."""
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import synth
from gpu_util import NAN_BITS, check_trimul_full, f32_bits

pytestmark = pytest.mark.gpu


def test_withheld_load_times_out_and_recovers(oracle_lib):
    shape = synth.TrimulShape(B=1, T=256, C=128, NH=2)
    qkv = synth.trimul_input(shape, seed=3).cuda()
    out = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")
    assert csa.get_status() == 0
    csa.set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        csa.debug_inject(True)
        csa.trimul_forward(out, qkv, shape.B, shape.T, shape.C, shape.NH)
        assert csa.get_status() == csa.CSA_ERR_TIMEOUT
        assert csa.get_status() == 0  # read-and-clear
    finally:
        csa.set_wait_limit_ns(0)
        csa.debug_inject(False)
    # the context still works and the next call is correct
    csa.trimul_forward(out, qkv, shape.B, shape.T, shape.C, shape.NH)
    assert csa.get_status() == 0
    ref = oracle_lib.trimul(synth.bf16_bits(qkv.cpu()).reshape(-1), shape.B, shape.T, shape.C,
                            shape.NH, 0)
    check_trimul_full(f32_bits(out), out.cpu().numpy(), ref, NAN_BITS, "after timeout")


def _timeout_then_recover(run, check):
    """run() once with the first hand-off withheld: CSA_ERR_TIMEOUT, read-and-clear;
    then run() again normally and check() its result."""
    assert csa.get_status() == 0
    csa.set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        csa.debug_inject(True)
        run()
        assert csa.get_status() == csa.CSA_ERR_TIMEOUT
        assert csa.get_status() == 0
    finally:
        csa.set_wait_limit_ns(0)
        csa.debug_inject(False)
    run()
    assert csa.get_status() == 0
    check()


def test_withheld_load_fp32_scores(oracle_lib):
    shape = synth.TrimulShape(B=1, T=200, C=128, NH=2)
    qkv = synth.trimul_input_f32(shape, seed=4)
    q = qkv.cuda()
    out = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")

    def check():
        ref = oracle_lib.trimul_f32(qkv.numpy().reshape(-1), shape.B, shape.T, shape.C,
                                    shape.NH, 0)
        check_trimul_full(f32_bits(out), out.cpu().numpy(), ref, NAN_BITS, "fp32 after timeout")

    _timeout_then_recover(lambda: csa.trimul_forward_f32(out, q, shape.B, shape.T, shape.C,
                                                         shape.NH), check)


def test_withheld_load_softmax(oracle_lib):
    shape = synth.TrimulShape(B=1, T=300, C=128, NH=2)
    qkv = synth.trimul_input(shape, seed=5)
    q = qkv.cuda()
    att = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")

    def check():
        from gpu_util import assert_close
        ref = oracle_lib.causal_softmax(synth.bf16_bits(qkv).reshape(-1), shape.B, shape.T,
                                        shape.C, shape.NH)
        assert_close(att.cpu().numpy(), ref, "softmax after timeout")

    _timeout_then_recover(lambda: csa.causal_softmax_forward(att, q, shape.B, shape.T, shape.C,
                                                             shape.NH), check)


@pytest.mark.parametrize("M,I,H,mode", [
    (960, 770, 768, csa.DENSE_FETCH_LOADERS),  # loader warps, 4-byte cp.async
    (300, 768, 512, csa.DENSE_FETCH_AUTO),     # TMA fetch
    (130, 771, 200, csa.DENSE_FETCH_LOADERS),  # loader warps, 2-byte loads
    (960, 770, 768, csa.DENSE_FETCH_AUTO),     # rows realigned into the workspace, then TMA
])
def test_withheld_hand_off_dense(oracle_lib, M, I, H, mode):
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=6)
    Xd, Wd = X.cuda(), W.cuda()
    Y = torch.empty((M, H), dtype=torch.float32, device="cuda")

    def check():
        from gpu_util import assert_close
        ref = oracle_lib.dense(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                               M, I, H)
        assert_close(Y.cpu().numpy(), ref, f"dense {M}x{I}x{H} after timeout")

    csa.set_dense_fetch(mode)
    try:
        _timeout_then_recover(lambda: csa.dense_xwt(Y, Xd, Wd, M, I, H), check)
    finally:
        csa.set_dense_fetch(csa.DENSE_FETCH_AUTO)


@pytest.mark.parametrize("M,I,H", [(6144, 768, 3072), (5000, 770, 3000)])
def test_withheld_hand_off_dense_pairs(oracle_lib, M, I, H):
    """A single call large enough to run as CTA pairs (TMA rows, and rows realigned into
    the workspace): both CTAs of the first pair withhold their first loads, the first
    CTA's MMA wait runs out, and the next call is correct on sampled rows."""
    import numpy as np
    from gpu_util import assert_close
    assert csa.dense_tiling(M, H, torch.cuda.get_device_properties(0).multi_processor_count)[1]
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=7)
    Xd, Wd = X.cuda(), W.cuda()
    Y = torch.empty((M, H), dtype=torch.float32, device="cuda")

    def check():
        rows = np.array([0, 255, 256, M // 2, M - 1])
        ref = oracle_lib.dense_rows(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                                    M, I, H, rows)
        assert_close(Y[torch.from_numpy(rows).cuda()].cpu().numpy(), ref,
                     f"dense {M}x{I}x{H} rows after timeout")
        assert bool(torch.all(torch.isfinite(Y)))

    _timeout_then_recover(lambda: csa.dense_xwt(Y, Xd, Wd, M, I, H), check)


def test_withheld_hand_off_dense_grouped(oracle_lib):
    """The grouped launch's TMA producer withholds its first load: the MMA warp's wait
    runs out, the status reports it, and the next call is correct."""
    I, H = 768, 512
    Ms = [200, 64, 333]
    Xs = [synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=M)[0] for M in Ms]
    W = synth.dense_input(synth.DenseShape(M=1, I=I, H=H), seed=3)[1]
    Xd = [X.cuda() for X in Xs]
    Wd = W.cuda()
    Ys = [torch.empty((M, H), dtype=torch.float32, device="cuda") for M in Ms]

    def check():
        from gpu_util import assert_close
        wbits = synth.bf16_bits(W).reshape(-1)
        for X, Y, M in zip(Xs, Ys, Ms):
            ref = oracle_lib.dense(synth.bf16_bits(X).reshape(-1), wbits, M, I, H)
            assert_close(Y.cpu().numpy(), ref, f"grouped M={M} after timeout")

    _timeout_then_recover(lambda: csa.dense_xwt_grouped(Ys, Xd, Wd, I, H), check)
