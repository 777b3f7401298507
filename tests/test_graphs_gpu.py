"""Every entry point captured in a CUDA graph and replayed: the replays give the same
bits as direct calls (GPU). A captured launch keeps the work-list counter slot it
was given at capture, so each replay relies on the previous one having left that
slot as it found it."""
import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import synth
from gpu_util import f32_bits, poisoned, trimul_case

pytestmark = pytest.mark.gpu

REPLAYS = 4


def _replayed_equals_direct(launch, outs):
    """`launch(stream)` writes `outs`; run it directly, then from a graph REPLAYS times
    (outputs poisoned before each replay), and compare bits."""
    launch(torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    want = [f32_bits(o).copy() for o in outs]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        launch(side)
    for _ in range(REPLAYS):
        for o in outs:
            o.view(torch.int32).fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert csa.get_status() == 0
        for o, w in zip(outs, want):
            assert np.array_equal(f32_bits(o), w)


@pytest.mark.parametrize("lower_only", [False, True])
def test_trimul_graph_replays(lower_only):
    shape, qkv = trimul_case(2, 300, 3, 64, seed=21)
    q = qkv.cuda()
    out = poisoned(shape.out_shape)
    _replayed_equals_direct(
        lambda s: csa.trimul_forward(out, q, 2, 300, shape.C, 3, lower_only=lower_only, stream=s),
        [out])


def test_trimul_f32_graph_replays():
    shape = synth.TrimulShape(B=1, T=260, C=2 * 64, NH=2)
    q = synth.trimul_input_f32(shape, seed=4).cuda()
    out = poisoned(shape.out_shape)
    _replayed_equals_direct(
        lambda s: csa.trimul_forward_f32(out, q, 1, 260, shape.C, 2, stream=s), [out])


def test_softmax_graph_replays():
    shape, qkv = trimul_case(1, 400, 2, 64, seed=22)
    q = qkv.cuda()
    att = poisoned(shape.out_shape)
    _replayed_equals_direct(
        lambda s: csa.causal_softmax_forward(att, q, 1, 400, shape.C, 2, stream=s), [att])


def test_batch_matmul_nt_graph_replays():
    X, W = synth.bmm_input(synth.BMM_NT_RAGGED, seed=3)
    bs = synth.BMM_NT_RAGGED
    Xd, Wd = X.cuda(), W.cuda()
    Y = poisoned((bs.batch, bs.T1, bs.T2))
    _replayed_equals_direct(
        lambda s: csa.batch_matmul_nt(Y, Xd, Wd, bs.batch, bs.T1, bs.T2, bs.D, stream=s), [Y])


def test_step_graph_replays():
    """A step of the score product, then the ragged dense layer (its rows realigned
    into a workspace inside its one launch), as one graph."""
    ts, ds = synth.TrimulShape(B=1, T=384, C=128, NH=2), synth.DenseShape(M=300, I=770, H=136)
    q = synth.trimul_input(ts, seed=5).cuda()
    X, W = synth.dense_input(ds, seed=6)
    Xd, Wd = X.cuda(), W.cuda()
    out = poisoned(ts.out_shape)
    Y = poisoned((ds.M, ds.H))

    def step(s):
        csa.trimul_forward(out, q, ts.B, ts.T, ts.C, ts.NH, stream=s)
        csa.dense_xwt(Y, Xd, Wd, ds.M, ds.I, ds.H, stream=s)

    _replayed_equals_direct(step, [out, Y])
