"""Work-list counter sets under concurrency (GPU). The score and softmax kernels
take positions from counter sets the library hands out per stream (and per
captured launch). A launch held back on one stream while 300 launches run on
another, launches on several streams released at once, and a CUDA graph replayed
beside direct launches must all give the oracle's result. Streams are held by a
host function (csa_debug_hold_stream), so nothing waits on the GPU."""
import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import _lib, synth
from gpu_util import check_trimul_full, f32_bits, poisoned, trimul_case

pytestmark = pytest.mark.gpu


def _scores_ref(oracle_lib, qkv, shape):
    return oracle_lib.trimul(synth.bf16_bits(qkv).reshape(-1), shape.B, shape.T, shape.C, shape.NH)


def _check_scores(out, ref, what):
    check_trimul_full(f32_bits(out), out.cpu().numpy().astype(np.float64), ref, 0x7FC00000, what)


def test_held_launch_and_300_launches_on_another_stream(oracle_lib):
    lib = _lib.load()
    sa, qa = trimul_case(1, 1000, 2, 64, seed=51)
    sb, qb = trimul_case(1, 700, 2, 64, seed=52)
    qa_d, qb_d = qa.cuda(), qb.cuda()
    out_a, att_a = poisoned(sa.out_shape), poisoned(sa.out_shape)
    out_b, att_b = poisoned(sb.out_shape), poisoned(sb.out_shape)
    A, B = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    assert lib.csa_debug_hold_stream(A.cuda_stream) == 0
    try:
        # held on A: a score launch (work list + fill pool) and a softmax launch
        csa.trimul_forward(out_a, qa_d, sa.B, sa.T, sa.C, sa.NH, stream=A)
        csa.causal_softmax_forward(att_a, qa_d, sa.B, sa.T, sa.C, sa.NH, stream=A)
        for i in range(300):
            csa.trimul_forward(out_b, qb_d, sb.B, sb.T, sb.C, sb.NH, stream=B)
            if i % 10 == 0:
                csa.causal_softmax_forward(att_b, qb_d, sb.B, sb.T, sb.C, sb.NH, stream=B)
    finally:
        lib.csa_debug_release_streams()
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    _check_scores(out_a, _scores_ref(oracle_lib, qa, sa), "held score launch")
    _check_scores(out_b, _scores_ref(oracle_lib, qb, sb), "after 300 launches")
    from gpu_util import assert_close
    for att, q, s, what in ((att_a, qa, sa, "held softmax"), (att_b, qb, sb, "softmax on B")):
        ref = oracle_lib.causal_softmax(synth.bf16_bits(q).reshape(-1), s.B, s.T, s.C, s.NH)
        assert_close(att.cpu().numpy(), ref, what)


def test_launches_on_eight_streams_released_together(oracle_lib):
    lib = _lib.load()
    cases = [trimul_case(1, 260 + 40 * k, 2, 64, seed=60 + k) for k in range(8)]
    streams = [torch.cuda.Stream() for _ in cases]
    outs = [poisoned(s.out_shape) for s, _ in cases]
    qs = [q.cuda() for _, q in cases]
    torch.cuda.synchronize()
    try:
        for st in streams:
            assert lib.csa_debug_hold_stream(st.cuda_stream) == 0
        for rep in range(5):
            for (s, _), q, out, st in zip(cases, qs, outs, streams):
                csa.trimul_forward(out, q, s.B, s.T, s.C, s.NH, stream=st)
    finally:
        lib.csa_debug_release_streams()
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    for k, ((s, q), out) in enumerate(zip(cases, outs)):
        _check_scores(out, _scores_ref(oracle_lib, q, s), f"stream {k}")


def test_graph_replayed_beside_direct_launches(oracle_lib):
    """A captured launch keeps a counter set of its own: replays of its graph on one
    stream run beside direct launches on another."""
    lib = _lib.load()
    sa, qa = trimul_case(1, 900, 2, 64, seed=71)
    sb, qb = trimul_case(1, 600, 2, 64, seed=72)
    qa_d, qb_d = qa.cuda(), qb.cuda()
    out_a, out_b = poisoned(sa.out_shape), poisoned(sb.out_shape)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        csa.trimul_forward(out_a, qa_d, sa.B, sa.T, sa.C, sa.NH, stream=side)
    A, B = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    out_a.view(torch.int32).fill_(-1)
    torch.cuda.synchronize()
    try:
        assert lib.csa_debug_hold_stream(A.cuda_stream) == 0
        assert lib.csa_debug_hold_stream(B.cuda_stream) == 0
        with torch.cuda.stream(A):
            for _ in range(20):
                g.replay()
        for _ in range(20):
            csa.trimul_forward(out_b, qb_d, sb.B, sb.T, sb.C, sb.NH, stream=B)
    finally:
        lib.csa_debug_release_streams()
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    _check_scores(out_a, _scores_ref(oracle_lib, qa, sa), "graph replays")
    _check_scores(out_b, _scores_ref(oracle_lib, qb, sb), "direct launches beside them")


def test_launches_from_four_host_threads(oracle_lib):
    """Four host threads, each on its own stream, launch score and softmax kernels at
    once: the counter sets are handed out under a lock, every result is the oracle's."""
    import threading
    cases = [trimul_case(1, 300 + 70 * k, 2, 64, seed=80 + k) for k in range(4)]
    qs = [q.cuda() for _, q in cases]
    outs = [poisoned(s.out_shape) for s, _ in cases]
    atts = [poisoned(s.out_shape) for s, _ in cases]
    streams = [torch.cuda.Stream() for _ in cases]
    errors = []

    def work(k):
        try:
            s, _ = cases[k]
            for _ in range(10):
                csa.trimul_forward(outs[k], qs[k], s.B, s.T, s.C, s.NH, stream=streams[k])
                csa.causal_softmax_forward(atts[k], qs[k], s.B, s.T, s.C, s.NH, stream=streams[k])
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    torch.cuda.synchronize()
    threads = [threading.Thread(target=work, args=(k,)) for k in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert csa.get_status() == 0
    from gpu_util import assert_close
    for k, ((s, q), out, att) in enumerate(zip(cases, outs, atts)):
        _check_scores(out, _scores_ref(oracle_lib, q, s), f"thread {k}")
        ref = oracle_lib.causal_softmax(synth.bf16_bits(q).reshape(-1), s.B, s.T, s.C, s.NH)
        assert_close(att.cpu().numpy(), ref, f"softmax thread {k}")
