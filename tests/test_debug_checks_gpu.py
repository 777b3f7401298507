"""The checking build (-DCSA_DEBUG: device-side checks of tile indices, ring
indices and TMEM column ranges) on small ragged cases of every entry point: no
check fails (status ok) and the results are bit-identical to the release
library's (GPU)."""
import ctypes

import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import _lib, build_lib, synth
from gpu_util import f32_bits, poisoned, trimul_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    lib = ctypes.CDLL(build_lib.build(debug=True))
    for name, (res, args) in _lib.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _same_and_clean(dbg, release_out, debug_out, what):
    torch.cuda.synchronize()
    assert csa.get_status() == 0, f"{what}: release status"
    assert dbg.csa_get_status(_stream()) == 0, f"{what}: a device check failed"
    assert np.array_equal(f32_bits(release_out), f32_bits(debug_out)), what


@pytest.mark.parametrize("B,T,NH,HS,flags", [(2, 300, 3, 64, 0), (1, 129, 2, 128, 0),
                                              (2, 300, 3, 64, 1), (1, 70, 1, 256, 0)])
def test_scores(dbg, B, T, NH, HS, flags):
    shape, qkv = trimul_case(B, T, NH, HS, seed=T + HS)
    q = qkv.cuda()
    a, b = poisoned(shape.out_shape), poisoned(shape.out_shape)
    csa.trimul_forward(a, q, B, T, shape.C, NH, lower_only=bool(flags))
    assert dbg.trimul_forward_ex(b.data_ptr(), q.data_ptr(), B, T, shape.C, NH, _lib.CSA_MASK_NAN,
                                 flags, _stream()) == 0
    _same_and_clean(dbg, a, b, f"scores {(B, T, NH, HS, flags)}")


@pytest.mark.parametrize("T,HS", [(260, 64), (200, 128)])
def test_scores_fp32(dbg, T, HS):
    shape = synth.TrimulShape(B=1, T=T, C=2 * HS, NH=2)
    q = synth.trimul_input_f32(shape, seed=T).cuda()
    a, b = poisoned(shape.out_shape), poisoned(shape.out_shape)
    csa.trimul_forward_f32(a, q, 1, T, shape.C, 2)
    assert dbg.trimul_forward_f32(b.data_ptr(), q.data_ptr(), 1, T, shape.C, 2,
                                  _lib.CSA_MASK_NAN, 0, _stream()) == 0
    _same_and_clean(dbg, a, b, f"fp32 scores T={T} HS={HS}")


def test_softmax(dbg):
    shape, qkv = trimul_case(2, 300, 2, 64, seed=31)
    q = qkv.cuda()
    a, b = poisoned(shape.out_shape), poisoned(shape.out_shape)
    csa.causal_softmax_forward(a, q, 2, 300, shape.C, 2)
    assert dbg.causal_softmax_forward(b.data_ptr(), q.data_ptr(), 2, 300, shape.C, 2,
                                      _stream()) == 0
    _same_and_clean(dbg, a, b, "softmax")


def test_batch_matmul_nt(dbg):
    bs = synth.BMM_NT_RAGGED
    X, W = synth.bmm_input(bs, seed=8)
    Xd, Wd = X.cuda(), W.cuda()
    a, b = poisoned((bs.batch, bs.T1, bs.T2)), poisoned((bs.batch, bs.T1, bs.T2))
    csa.batch_matmul_nt(a, Xd, Wd, bs.batch, bs.T1, bs.T2, bs.D)
    assert dbg.batch_matmul_nt(b.data_ptr(), Xd.data_ptr(), Wd.data_ptr(), bs.batch, bs.T1,
                               bs.T2, bs.D, _stream()) == 0
    _same_and_clean(dbg, a, b, "batched NT")


# (the last two run as CTA pairs: an odd number of m-tiles with H % 4 != 0, and a ragged
# last k-block)
@pytest.mark.parametrize("M,I,H", [(960, 770, 768), (300, 768, 136), (2049, 256, 3072),
                                   (12345, 768, 3071), (6500, 136, 4100)])
def test_dense(dbg, M, I, H):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert csa.dense_tiling(M, H, sms)[1] == (M > 5000)
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=M)
    Xd, Wd = X.cuda(), W.cuda()
    a, b = poisoned((M, H)), poisoned((M, H))
    csa.dense_xwt(a, Xd, Wd, M, I, H)
    assert dbg.dense_xwt_ex(b.data_ptr(), Xd.data_ptr(), Wd.data_ptr(), M, I, H, _stream()) == 0
    _same_and_clean(dbg, a, b, f"dense {(M, I, H)}")


def test_dense_grouped(dbg):
    xs, W = synth.dense_sweep_inputs(seed=0)
    H, I = W.shape
    Wd = W.cuda()
    Xd = [X.cuda() for X in xs[:9]]  # an odd number of m-tiles in total: a phantom half-pair
    a = [poisoned((X.shape[0], H)) for X in Xd]
    b = [poisoned((X.shape[0], H)) for X in Xd]
    csa.dense_xwt_grouped(a, Xd, Wd, I, H)
    n = len(Xd)
    ys = (ctypes.c_void_p * n)(*[y.data_ptr() for y in b])
    xp = (ctypes.c_void_p * n)(*[x.data_ptr() for x in Xd])
    ms = (ctypes.c_int * n)(*[x.shape[0] for x in Xd])
    assert dbg.dense_xwt_grouped(ctypes.addressof(ys), ctypes.addressof(xp), Wd.data_ptr(),
                                 ctypes.addressof(ms), n, I, H, _stream()) == 0
    torch.cuda.synchronize()
    for g in range(n):
        _same_and_clean(dbg, a[g], b[g], f"grouped problem {g}")


def test_noalloc_clears_scratch_left_mid_list(dbg):
    """trimul_forward_noalloc clears its fixed scratch before each kernel: with the
    counters left non-zero (as by a launch that stopped mid-list; the checking build
    can plant that), the call still writes every tile, the release library's bits."""
    fill = dbg.csa_debug_noalloc_scratch_fill
    fill.restype, fill.argtypes = ctypes.c_int, [ctypes.c_uint32]
    shape, qkv = trimul_case(2, 300, 3, 64, seed=41)
    q = qkv.cuda()
    a = poisoned(shape.out_shape)
    csa.trimul_forward(a, q, 2, 300, shape.C, 3)
    for value in (7, 0x00FFFFFF):
        assert fill(value) == 0
        b = poisoned(shape.out_shape)
        assert dbg.trimul_forward_noalloc(b.data_ptr(), q.data_ptr(), 2, 300, shape.C, 3,
                                          _lib.CSA_MASK_NAN, 0, _stream()) == 0
        _same_and_clean(dbg, a, b, f"noalloc after scratch filled with {value:#x}")
