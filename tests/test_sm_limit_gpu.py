"""Per-stream SM limits (GPU). A limit changes the grid and the tiling of every
kernel of the library, never its bits: each call under a limit must equal the same
call without one, and calls on two limited streams running side by side must equal
the same calls one after another. The oracle pins the unlimited results."""
import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import synth
from gpu_util import check_trimul_full, f32_bits, poisoned, trimul_case

pytestmark = pytest.mark.gpu

LIMITS = [1, 2, 7, 56, 151]


@pytest.fixture
def limited_stream():
    s = torch.cuda.Stream()
    yield s
    csa.set_stream_sm_limit(s, 0)


def _same(a, b, what):
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    assert np.array_equal(f32_bits(a), f32_bits(b)), what


def test_scores_under_limits(oracle_lib, limited_stream):
    shape, qkv = trimul_case(2, 777, 3, 64, seed=61)
    q = qkv.cuda()
    ref = oracle_lib.trimul(synth.bf16_bits(qkv).reshape(-1), shape.B, shape.T, shape.C, shape.NH)
    base = poisoned(shape.out_shape)
    csa.trimul_forward(base, q, shape.B, shape.T, shape.C, shape.NH)
    torch.cuda.synchronize()
    check_trimul_full(f32_bits(base), base.cpu().numpy().astype(np.float64), ref, 0x7FC00000,
                      "unlimited")
    for lim in LIMITS:
        csa.set_stream_sm_limit(limited_stream, lim)
        assert csa.get_stream_sm_limit(limited_stream) == lim
        for lower_only in (False, True):
            out = poisoned(shape.out_shape)
            if lower_only:
                ref_lo = poisoned(shape.out_shape)
                csa.trimul_forward(ref_lo, q, shape.B, shape.T, shape.C, shape.NH,
                                   lower_only=True)
            csa.trimul_forward(out, q, shape.B, shape.T, shape.C, shape.NH,
                               lower_only=lower_only, stream=limited_stream)
            _same(out, ref_lo if lower_only else base, f"scores, limit {lim}, lower {lower_only}")


def test_softmax_and_batched_nt_under_limits(limited_stream):
    shape, qkv = trimul_case(1, 515, 2, 64, seed=62)
    q = qkv.cuda()
    base = poisoned(shape.out_shape)
    csa.causal_softmax_forward(base, q, shape.B, shape.T, shape.C, shape.NH)
    X = torch.randn(3, 200, 64, device="cuda").to(torch.bfloat16)
    W = torch.randn(3, 300, 64, device="cuda").to(torch.bfloat16)
    ybase = poisoned((3, 200, 300))
    csa.batch_matmul_nt(ybase, X, W, 3, 200, 300, 64)
    for lim in LIMITS:
        csa.set_stream_sm_limit(limited_stream, lim)
        att = poisoned(shape.out_shape)
        csa.causal_softmax_forward(att, q, shape.B, shape.T, shape.C, shape.NH,
                                   stream=limited_stream)
        _same(att, base, f"softmax, limit {lim}")
        y = poisoned((3, 200, 300))
        csa.batch_matmul_nt(y, X, W, 3, 200, 300, 64, stream=limited_stream)
        _same(y, ybase, f"batch_matmul_nt, limit {lim}")


@pytest.mark.parametrize("M,I,H", [(5000, 770, 3000), (12345, 768, 3071), (960, 770, 768)])
def test_dense_under_limits(oracle_lib, limited_stream, M, I, H):
    """Large calls (CTA pairs without a limit; a limit of 1 leaves no pair) and the
    ragged case, through dense_xwt (workspace allocated on the call's stream)."""
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=M)
    Xd, Wd = X.cuda(), W.cuda()
    base = poisoned((M, H))
    csa.dense_xwt(base, Xd, Wd, M, I, H)
    torch.cuda.synchronize()
    rows = np.array([0, M // 2, M - 1])
    ref = oracle_lib.dense_rows(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                                M, I, H, rows)
    got = base[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref) / (1 + np.abs(ref))) < 1e-5
    for lim in LIMITS:
        csa.set_stream_sm_limit(limited_stream, lim)
        Y = poisoned((M, H))
        csa.dense_xwt(Y, Xd, Wd, M, I, H, stream=limited_stream)
        _same(Y, base, f"dense {(M, I, H)}, limit {lim}")


def test_grouped_under_limits(limited_stream):
    xs, W = synth.dense_sweep_inputs(seed=0)
    Wd = W.cuda()
    Xs = [x.cuda() for x in xs[:12]]
    H, I = W.shape
    base = [poisoned((x.shape[0], H)) for x in Xs]
    csa.dense_xwt_grouped(base, Xs, Wd, I, H)
    for lim in LIMITS:
        csa.set_stream_sm_limit(limited_stream, lim)
        Ys = [poisoned((x.shape[0], H)) for x in Xs]
        csa.dense_xwt_grouped(Ys, Xs, Wd, I, H, stream=limited_stream)
        for g, (a, b) in enumerate(zip(Ys, base)):
            _same(a, b, f"grouped problem {g}, limit {lim}")


def test_side_by_side_streams_equal_one_after_another():
    """The default bench step's schedule at a smaller size: the dense calls on a
    stream limited to 56 SMs, launched first, and the score kernel on a stream with
    no limit, repeated; every output equals the sequential calls' bits."""
    shape, qkv = trimul_case(2, 2048, 8, 128, seed=63)
    q = qkv.cuda()
    xs, W = synth.dense_sweep_inputs(seed=1)
    Wd = W.cuda()
    Xs = [x.cuda() for x in xs]
    H, I = W.shape
    Xr, Wr = (t.cuda() for t in synth.dense_input(synth.DENSE_RAGGED, seed=0))
    R = synth.DENSE_RAGGED

    def run(dense_stream, score_stream):
        out = poisoned(shape.out_shape)
        Ys = [poisoned((x.shape[0], H)) for x in Xs]
        Yr = poisoned((R.M, R.H))
        main = torch.cuda.current_stream()
        dense_stream.wait_stream(main)
        score_stream.wait_stream(main)
        csa.dense_xwt_grouped(Ys, Xs, Wd, I, H, stream=dense_stream)
        csa.dense_xwt(Yr, Xr, Wr, R.M, R.I, R.H, stream=dense_stream)
        csa.trimul_forward(out, q, shape.B, shape.T, shape.C, shape.NH, stream=score_stream)
        main.wait_stream(dense_stream)
        main.wait_stream(score_stream)
        return [out, Yr] + Ys

    main = torch.cuda.current_stream()
    base = run(main, main)
    sd, ss = torch.cuda.Stream(), torch.cuda.Stream()
    csa.set_stream_sm_limit(sd, 56)
    try:
        for rep in range(5):
            outs = run(sd, ss)
            for k, (a, b) in enumerate(zip(outs, base)):
                _same(a, b, f"output {k}, repetition {rep}")
    finally:
        csa.set_stream_sm_limit(sd, 0)


def test_side_by_side_streams_in_a_cuda_graph():
    """The same schedule captured once into a CUDA graph (the bench's form of the default
    step: a fork from the capturing stream into the two limited streams and a join) and
    replayed: every replay equals the calls made one after another."""
    shape, qkv = trimul_case(1, 1536, 4, 64, seed=64)
    q = qkv.cuda()
    xs, W = synth.dense_sweep_inputs(seed=2)
    Wd = W.cuda()
    Xs = [x.cuda() for x in xs[:16]]
    H, I = W.shape
    out = poisoned(shape.out_shape)
    Ys = [poisoned((x.shape[0], H)) for x in Xs]
    plan = csa.DenseGroupedPlan(Ys, Xs, Wd, I, H)
    main = torch.cuda.current_stream()
    plan(main)
    csa.trimul_forward(out, q, shape.B, shape.T, shape.C, shape.NH, stream=main)
    torch.cuda.synchronize()
    base = [out.clone()] + [y.clone() for y in Ys]

    sd, ss, cap = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    csa.set_stream_sm_limit(sd, 56)
    try:
        graph = torch.cuda.CUDAGraph()
        cap.wait_stream(main)
        with torch.cuda.graph(graph, stream=cap):
            sd.wait_stream(cap)
            ss.wait_stream(cap)
            plan(sd)
            csa.trimul_forward(out, q, shape.B, shape.T, shape.C, shape.NH, stream=ss)
            cap.wait_stream(sd)
            cap.wait_stream(ss)
        for rep in range(3):
            out.view(torch.int32).fill_(-1)
            for y in Ys:
                y.view(torch.int32).fill_(-1)
            graph.replay()
            for k, (a, b) in enumerate(zip([out] + Ys, base)):
                _same(a, b, f"output {k}, replay {rep}")
    finally:
        csa.set_stream_sm_limit(sd, 0)
