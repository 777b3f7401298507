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
