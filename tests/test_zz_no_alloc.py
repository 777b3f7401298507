"""trimul_forward_noalloc, the entry point for callers that may not allocate
device memory (a memory manager that forbids allocations after start-up, a
region that cannot take cudaFree's device-wide synchronisation, a plug-in host
that only hands out buffers). It keeps its scratch in a fixed device array
instead, and must produce what trimul_forward_ex produces.

Each case calls it twice in a row through the C ABI: the second call starts
from whatever scratch the first call left behind, so both must match the
existing entry point within the tolerance the parity tests use. This file is
named to be collected last.
"""
import pytest
import torch

from causal_attention_score_gb300 import _lib, synth
from gpu_util import NAN_BITS, TOL

pytestmark = pytest.mark.gpu


def _compare(got: torch.Tensor, want: torch.Tensor, what: str) -> None:
    gb, wb = got.view(torch.int32), want.view(torch.int32)
    masked = torch.isnan(want) | torch.isinf(want)
    assert torch.equal(gb[masked], wb[masked]), f"{what}: mask bits differ"
    g, w = got[~masked].double(), want[~masked].double()
    assert bool(torch.all(torch.isfinite(g))), f"{what}: non-finite values"
    err = ((g - w).abs() / (1.0 + w.abs())).max().item() if g.numel() else 0.0
    assert err <= TOL, f"{what}: max scaled error {err}"


@pytest.mark.parametrize("B,T,NH,HS,flags", [
    (2, 300, 3, 64, 0),                       # ragged T, full output
    (2, 300, 3, 64, _lib.CSA_TRIMUL_LOWER_ONLY),
    (8, 1024, 12, 64, 0),                     # the GPT-2-small shape
])
def test_noalloc_matches_trimul_forward_ex_twice(B, T, NH, HS, flags):
    lib = _lib.load()
    shape = synth.TrimulShape(B=B, T=T, C=NH * HS, NH=NH)
    qkv = synth.trimul_input(shape, seed=B + T).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    want = torch.empty(shape.out_shape, dtype=torch.float32, device="cuda")
    want.view(torch.int32).fill_(-1)
    assert lib.trimul_forward_ex(want.data_ptr(), qkv.data_ptr(), B, T, shape.C, NH, NAN_BITS,
                                 flags, stream) == 0
    for call in range(2):
        got = torch.empty_like(want)
        got.view(torch.int32).fill_(-1)
        rc = lib.trimul_forward_noalloc(got.data_ptr(), qkv.data_ptr(), B, T, shape.C, NH,
                                        NAN_BITS, flags, stream)
        assert rc == 0, lib.csa_last_error()
        assert lib.csa_get_status(stream) == 0
        _compare(got, want, f"call {call}")
