"""Parity of the CUDA ragged dense layer Y = X W^T against the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import causal_attention_score_gb300 as csa
from causal_attention_score_gb300 import synth
from gpu_util import assert_close, f32_bits, poisoned

pytestmark = pytest.mark.gpu

# (M, I, H): the ragged case (M % 128 != 0, I % 4 != 0), the page's H = 2304, TMA-able
# and non-TMA I, odd I (2-byte loads), H % 4 != 0 (plain stores), tiny and tile-edge sizes.
SHAPES = [
    (960, 770, 768),
    (960, 770, 2304),
    (1, 8, 1),
    (17, 770, 768),
    (130, 776, 200),
    (128, 64, 128),
    (129, 65, 129),
    (33, 21, 7),
    (7, 300, 5),
    (64, 768, 3072),
    (300, 1000, 770),
    (257, 129, 255),
    # bulk + realign fetch (I even, rows not 16-byte multiples), incl. rows shorter
    # than the 144-byte copy window and arrays whose size is not a multiple of 16
    (33, 10, 17),
    (5, 2, 3),
    (7, 10, 9),
    (200, 130, 300),
    (131, 258, 129),
    (1024, 770, 1024),
]


def _run(X, W):
    M, I = X.shape
    H = W.shape[0]
    Y = poisoned((M, H))
    csa.dense_xwt(Y, X.cuda(), W.cuda(), M, I, H)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    return Y


@pytest.mark.parametrize("M,I,H", SHAPES)
def test_dense_parity(oracle_lib, M, I, H):
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=M + I + H)
    ref = oracle_lib.dense(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1), M, I, H)
    Y = _run(X, W)
    assert_close(Y.cpu().numpy(), ref, f"dense{(M, I, H)}")


def test_dense_ragged_case(oracle_lib):
    """The ragged case: X [960, 770], W [768, 770], seed 0, via the allocating helper."""
    s = synth.DENSE_RAGGED
    X, W = synth.dense_input(s, seed=0)
    ref = oracle_lib.dense(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                           s.M, s.I, s.H)
    Y = csa.dense(X.cuda(), W.cuda())
    torch.cuda.synchronize()
    assert_close(Y.cpu().numpy(), ref, "dense ragged")


@pytest.mark.parametrize("M,I,H", [(960, 770, 768), (200, 776, 130), (31, 33, 29)])
def test_dense_integer_inputs_bit_exact(oracle_lib, M, I, H):
    rng = np.random.default_rng(M)
    X = torch.from_numpy(rng.integers(-4, 5, size=(M, I)).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy(rng.integers(-4, 5, size=(H, I)).astype(np.float32)).to(torch.bfloat16)
    ref = oracle_lib.dense(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1), M, I, H)
    Y = _run(X, W)
    assert np.array_equal(Y.cpu().numpy().astype(np.float64), ref)


def test_dense_row_independence():
    """One row computed alone equals that row of the full product (no leakage
    through the zero-filled tile padding)."""
    X, W = synth.dense_input(synth.DenseShape(M=333, I=770, H=768), seed=5)
    Y = _run(X, W)
    for r in (0, 127, 128, 332):
        y1 = _run(X[r:r + 1].contiguous(), W)
        assert torch.equal(y1[0], Y[r])


def test_dense_sweep(oracle_lib):
    """All 32 calls of the dynamic-shape sweep (M = 16*T, T ~ U{1..128}, I=768, H=3072),
    on sampled rows of each call."""
    xs, W = synth.dense_sweep_inputs(seed=0)
    Wd = W.cuda()
    wbits = synth.bf16_bits(W).reshape(-1)
    H, I = W.shape
    rng = np.random.default_rng(0)
    for i, X in enumerate(xs):
        M = X.shape[0]
        Y = poisoned((M, H))
        csa.dense_xwt(Y, X.cuda(), Wd, M, I, H)
        torch.cuda.synchronize()
        rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, size=6)]))
        ref = oracle_lib.dense_rows(synth.bf16_bits(X).reshape(-1), wbits, M, I, H, rows)
        assert_close(Y[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, f"sweep call {i} M={M}")
        assert bool(torch.all(torch.isfinite(Y)))


# Single calls that run as CTA pairs on a 152-SM GB300 (the tiling model, counting pairs
# of m-tiles over 76 clusters, costs no more than single CTAs and gives each cluster
# three tiles or more): realigned rows (I = 770) with H not a multiple of the tile
# width; an odd number of m-tiles (the last pair's second half lies past M) with
# H % 4 != 0 (plain stores); a single k-block; a ragged last k-block (I = 136); and a
# shape that takes single CTAs, for contrast.
PAIR_SHAPES = [(5000, 770, 3000, True), (12345, 768, 3071, True), (30000, 64, 2304, True),
               (6500, 136, 4100, True), (2049, 768, 3072, False)]


@pytest.mark.parametrize("M,I,H,pairs", PAIR_SHAPES)
def test_dense_large_call_matches_512_row_calls_and_oracle(oracle_lib, M, I, H, pairs):
    """Every row of a large call (CTA pairs, but for the last shape) equals, bit for bit,
    the same row from calls of 512 rows (single CTAs: the same products summed in the
    same k order), and sampled rows match the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert csa.dense_tiling(M, H, sms)[1] == pairs
    assert not csa.dense_tiling(512, H, sms)[1]
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=M + H)
    Xd, Wd = X.cuda(), W.cuda()
    Y = poisoned((M, H))
    csa.dense_xwt(Y, Xd, Wd, M, I, H)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    assert bool(torch.all(torch.isfinite(Y)))
    for r0 in range(0, M, 512):
        n = min(512, M - r0)
        Ys = poisoned((n, H))
        csa.dense_xwt(Ys, Xd[r0:r0 + n], Wd, n, I, H)
        torch.cuda.synchronize()
        assert torch.equal(Y[r0:r0 + n], Ys), f"rows {r0}..{r0 + n} of {(M, I, H)}"
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([[0, M - 1, (M - 1) // 256 * 256], rng.integers(0, M, size=6)]))
    ref = oracle_lib.dense_rows(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                                M, I, H, rows)
    assert_close(Y[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, f"dense{(M, I, H)} rows")


@pytest.fixture(params=["auto", "loaders"])
def fetch_mode(request):
    """Both fetch paths for rows no tensor map can describe: the rows realigned into
    the workspace + TMA (default) and the loader warps (workspace unused)."""
    mode = csa.DENSE_FETCH_AUTO if request.param == "auto" else csa.DENSE_FETCH_LOADERS
    csa.set_dense_fetch(mode)
    yield request.param
    csa.set_dense_fetch(csa.DENSE_FETCH_AUTO)


# Shapes whose rows no tensor map can describe (I * 2 % 16 != 0): even and odd I,
# rows shorter than one 16-byte chunk, ragged tiles on every axis.
MISALIGNED_ROWS = [(960, 770, 768), (17, 770, 768), (129, 65, 129), (33, 21, 7), (5, 2, 3),
                   (7, 10, 9), (131, 258, 129), (300, 1002, 770), (1, 1, 1)]


@pytest.mark.parametrize("M,I,H", MISALIGNED_ROWS)
def test_dense_fetch_paths(oracle_lib, fetch_mode, M, I, H):
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=3 * M + I)
    ref = oracle_lib.dense(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1), M, I, H)
    Y = _run(X, W)
    assert_close(Y.cpu().numpy(), ref, f"dense{(M, I, H)} fetch={fetch_mode}")


@pytest.mark.parametrize("M,I,H", [(960, 770, 768), (257, 129, 255), (40, 1000, 3072)])
def test_dense_fetch_paths_bit_identical(M, I, H):
    """The realigned copy and the loader warps feed the same tiles in the same
    order: the two results are equal bit for bit."""
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=11)
    try:
        csa.set_dense_fetch(csa.DENSE_FETCH_LOADERS)
        y_loaders = _run(X, W)
    finally:
        csa.set_dense_fetch(csa.DENSE_FETCH_AUTO)
    y_auto = _run(X, W)
    assert np.array_equal(f32_bits(y_auto), f32_bits(y_loaders))


def test_dense_fetch_mode_rejects_unknown():
    with pytest.raises(csa.CsaError):
        csa.set_dense_fetch(7)


def test_dense_realigned_on_streams_and_graph(oracle_lib):
    """The binding's workspace is stream-ordered: calls on two streams at once, and
    the call captured in a CUDA graph and replayed, give the oracle's result."""
    M, I, H = 300, 770, 512
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=21)
    ref = oracle_lib.dense(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1), M, I, H)
    Xd, Wd = X.cuda(), W.cuda()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ys = [poisoned((M, H)), poisoned((M, H))]
    torch.cuda.synchronize()
    for _ in range(4):
        for st, y in zip(streams, ys):
            csa.dense_xwt(y, Xd, Wd, M, I, H, stream=st)
    torch.cuda.synchronize()
    for y in ys:
        assert_close(y.cpu().numpy(), ref, "dense on two streams")
    side = torch.cuda.Stream()
    yg = poisoned((M, H))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        csa.dense_xwt(yg, Xd, Wd, M, I, H, stream=side)
    for _ in range(3):
        yg.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    assert_close(yg.cpu().numpy(), ref, "dense replayed from a graph")


@pytest.mark.parametrize("offset", [1, 2])
def test_dense_misaligned_views(oracle_lib, fetch_mode, offset):
    """X and W views starting 2 or 4 bytes into their storage: not 16-byte aligned,
    so they are read 2 bytes or 4 bytes at a time (by the realigning copy or by
    the loader warps)."""
    M, I, H = 130, 770, 70
    Xb, Wb = synth.dense_input(synth.DenseShape(M=M, I=I + offset, H=H), seed=9)
    Xf = Xb.reshape(-1)[offset:offset + M * I].reshape(M, I)
    Wf = Wb.reshape(-1)[offset:offset + H * I].reshape(H, I)
    Xd = Xb.reshape(-1).cuda()[offset:offset + M * I]
    Wd = Wb.reshape(-1).cuda()[offset:offset + H * I]
    assert Xd.data_ptr() % 16 != 0
    ref = oracle_lib.dense(synth.bf16_bits(Xf.contiguous()).reshape(-1),
                           synth.bf16_bits(Wf.contiguous()).reshape(-1), M, I, H)
    Y = poisoned((M, H))
    csa.dense_xwt(Y, Xd, Wd, M, I, H)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    assert_close(Y.cpu().numpy(), ref, f"misaligned by {2 * offset} bytes")


def _ws_call(Y, X, W, ws, stream=None):
    M, I = X.shape
    H = W.shape[0]
    csa.dense_xwt_ws(Y, X, W, M, I, H, ws, stream=stream)


def test_dense_ws_ragged_case_against_oracle(oracle_lib):
    """dense_xwt_ws with a caller workspace on the ragged case X [960, 770], W [768, 770]
    (seed 0): the rows realigned into the workspace, then the TMA product."""
    s = synth.DENSE_RAGGED
    X, W = synth.dense_input(s, seed=0)
    ref = oracle_lib.dense(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                           s.M, s.I, s.H)
    Xd, Wd = X.cuda(), W.cuda()
    n = csa.dense_workspace_size(Xd, Wd, s.M, s.I, s.H)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    Y = poisoned((s.M, s.H))
    _ws_call(Y, Xd, Wd, ws)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    assert_close(Y.cpu().numpy(), ref, "dense_xwt_ws ragged")


@pytest.mark.parametrize("M,I,H", [(960, 770, 768), (1024, 770, 1024), (4000, 770, 768),
                                   (300, 1002, 770), (129, 65, 129)])
def test_dense_ws_garbage_and_reused_workspace(oracle_lib, M, I, H):
    """The workspace needs no clearing: filled with garbage, or holding a previous
    call's copy (of this shape or another), every call gives the oracle's result,
    and repeated calls the same bits. Shapes with more tiles than SMs make a CTA
    compute several tiles in turn."""
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=M + 7 * I)
    ref = oracle_lib.dense(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1), M, I, H)
    Xd, Wd = X.cuda(), W.cuda()
    n = csa.dense_workspace_size(Xd, Wd, M, I, H)
    ws = torch.empty(n + 4096, dtype=torch.uint8, device="cuda")
    ws.random_(0, 256, generator=torch.Generator(device="cuda").manual_seed(M))
    first = None
    for k in range(3):
        if k == 2:
            # a different shape through the same workspace, then this one again
            X2, W2 = synth.dense_input(synth.DenseShape(M=33, I=I, H=65), seed=1)
            Y2 = poisoned((33, 65))
            _ws_call(Y2, X2.cuda(), W2.cuda(), ws)
        Y = poisoned((M, H))
        _ws_call(Y, Xd, Wd, ws)
        torch.cuda.synchronize()
        assert csa.get_status() == 0
        assert_close(Y.cpu().numpy(), ref, f"dense_xwt_ws{(M, I, H)} call {k}")
        if first is None:
            first = f32_bits(Y)
        else:
            assert np.array_equal(f32_bits(Y), first), "repeated calls differ in bits"


def test_dense_ws_matches_workspace_free_call_bits():
    """dense_xwt_ex without workspace (loader warps) and dense_xwt_ws (realigned copy
    + TMA) on the same operands: the same tiles summed in the same order, the same
    bits."""
    M, I, H = 960, 770, 768
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=4)
    Xd, Wd = X.cuda(), W.cuda()
    Ya, Yb = poisoned((M, H)), poisoned((M, H))
    from causal_attention_score_gb300 import _lib
    rc = _lib.load().dense_xwt_ex(Ya.data_ptr(), Xd.data_ptr(), Wd.data_ptr(), M, I, H,
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    ws = torch.empty(csa.dense_workspace_size(Xd, Wd, M, I, H), dtype=torch.uint8,
                     device="cuda")
    _ws_call(Yb, Xd, Wd, ws)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    assert np.array_equal(f32_bits(Ya), f32_bits(Yb))


def test_dense_calls_leave_device_memory_unchanged():
    """No call allocates: after a first call of each form (which loads the kernels),
    further calls leave the device's free memory exactly where it was."""
    M, I, H = 960, 770, 768
    X, W = synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=2)
    Xd, Wd = X.cuda(), W.cuda()
    Xs, Ws = synth.dense_input(synth.DenseShape(M=200, I=768, H=512), seed=3)
    Xs, Ws = Xs.cuda(), Ws.cuda()
    ws = torch.empty(csa.dense_workspace_size(Xd, Wd, M, I, H), dtype=torch.uint8,
                     device="cuda")
    Y, Ys = torch.empty((M, H), device="cuda"), torch.empty((200, 512), device="cuda")
    from causal_attention_score_gb300 import _lib
    lib = _lib.load()
    st = torch.cuda.current_stream().cuda_stream

    def calls():
        assert lib.dense_xwt_ex(Y.data_ptr(), Xd.data_ptr(), Wd.data_ptr(), M, I, H, st) == 0
        _ws_call(Y, Xd, Wd, ws)
        assert lib.dense_xwt_ex(Ys.data_ptr(), Xs.data_ptr(), Ws.data_ptr(), 200, 768, 512,
                                st) == 0

    calls()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(20):
        calls()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert csa.get_status() == 0


def _grouped_vs_single(Xs, W, I, H, what):
    """dense_xwt_grouped against one dense_xwt per problem: equal bit for bit (same
    k-order per element whatever the tile width)."""
    Wd = W.cuda()
    Xd = [X.cuda() for X in Xs]
    Yg = [poisoned((X.shape[0], H)) for X in Xs]
    csa.dense_xwt_grouped(Yg, Xd, Wd, I, H)
    Ys = [poisoned((X.shape[0], H)) for X in Xs]
    for Y, X in zip(Ys, Xd):
        csa.dense_xwt(Y, X, Wd, X.shape[0], I, H)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    for g, (a, b) in enumerate(zip(Yg, Ys)):
        assert np.array_equal(f32_bits(a), f32_bits(b)), f"{what}: problem {g}"
    return Yg


def test_dense_grouped_sweep(oracle_lib):
    """The dynamic-shape sweep's 32 problems in one grouped call: equal to 32 separate
    calls, and sampled rows of each against the oracle."""
    xs, W = synth.dense_sweep_inputs(seed=0)
    H, I = W.shape
    Yg = _grouped_vs_single(xs, W, I, H, "sweep")
    wbits = synth.bf16_bits(W).reshape(-1)
    rng = np.random.default_rng(11)
    for g in (0, 5, 17, 31):
        X = xs[g]
        M = X.shape[0]
        rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, size=4)]))
        ref = oracle_lib.dense_rows(synth.bf16_bits(X).reshape(-1), wbits, M, I, H, rows)
        assert_close(Yg[g][torch.from_numpy(rows).cuda()].cpu().numpy(), ref, f"grouped {g}")


@pytest.mark.parametrize("I,H", [(768, 200), (64, 130), (128, 3072), (770, 96)])
def test_dense_grouped_mixed_rows(oracle_lib, I, H):
    """Row counts on both sides of the 128-row tile, one row, and a multi-wave problem;
    H = 130 writes Y with plain stores; I = 770 rows are not TMA-describable, so the
    group runs as separate calls."""
    Ms = [1, 127, 128, 129, 300, 2049]
    Xs = [synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=M)[0] for M in Ms]
    W = synth.dense_input(synth.DenseShape(M=1, I=I, H=H), seed=99)[1]
    Yg = _grouped_vs_single(Xs, W, I, H, f"mixed I={I} H={H}")
    wbits = synth.bf16_bits(W).reshape(-1)
    for g in (0, 3, 5):
        ref = oracle_lib.dense(synth.bf16_bits(Xs[g]).reshape(-1), wbits, Ms[g], I, H)
        assert_close(Yg[g].cpu().numpy(), ref, f"grouped M={Ms[g]}")


def test_dense_grouped_more_than_one_launch():
    """100 problems: more than one launch's worth (48 each)."""
    rng = np.random.default_rng(5)
    I, H = 256, 192
    Ms = rng.integers(1, 400, size=100).tolist()
    Xs = [synth.dense_input(synth.DenseShape(M=M, I=I, H=H), seed=i)[0] for i, M in enumerate(Ms)]
    W = synth.dense_input(synth.DenseShape(M=1, I=I, H=H), seed=7)[1]
    _grouped_vs_single(Xs, W, I, H, "100 problems")


def test_dense_grouped_graph_replay():
    xs, W = synth.dense_sweep_inputs(seed=0)
    H, I = W.shape
    Wd = W.cuda()
    Xd = [X.cuda() for X in xs[:8]]
    ref = [poisoned((X.shape[0], H)) for X in Xd]
    csa.dense_xwt_grouped(ref, Xd, Wd, I, H)
    Yg = [poisoned((X.shape[0], H)) for X in Xd]
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        csa.dense_xwt_grouped(Yg, Xd, Wd, I, H, stream=side)
    for _ in range(3):
        for Y in Yg:
            Y.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    for a, b in zip(Yg, ref):
        assert np.array_equal(f32_bits(a), f32_bits(b))


def test_dense_grouped_plan_repeats_and_notices_new_storage():
    """A DenseGroupedPlan launches the same products as dense_xwt_grouped, call after
    call, and refuses to run once one of its tensors has new storage."""
    xs, W = synth.dense_sweep_inputs(seed=0)
    H, I = W.shape
    Wd = W.cuda()
    Xd = [X.cuda() for X in xs[:6]]
    ref = [poisoned((X.shape[0], H)) for X in Xd]
    csa.dense_xwt_grouped(ref, Xd, Wd, I, H)
    Yp = [poisoned((X.shape[0], H)) for X in Xd]
    plan = csa.DenseGroupedPlan(Yp, Xd, Wd, I, H)
    for _ in range(3):
        for Y in Yp:
            Y.fill_(float("nan"))
        plan()
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    for a, b in zip(Yp, ref):
        assert np.array_equal(f32_bits(a), f32_bits(b))
    Yp[2].set_(torch.empty_like(Yp[2]))  # the tensor now points at other memory
    with pytest.raises(ValueError):
        plan()


@pytest.mark.parametrize("I,H,offset", [(770, 768, 0), (771, 200, 0), (768, 300, 1)])
def test_dense_grouped_realigned_rows(oracle_lib, I, H, offset):
    """A grouped call whose rows no tensor map can describe (I = 770 and 771, or views
    starting 2 bytes into their storage) runs as one copy into the plan's workspace and
    one grouped launch: the same bits as one dense_xwt per problem, and the oracle's
    values on sampled rows."""
    Ms = [45, 300, 17, 128, 1000, 3]
    rng = np.random.default_rng(I + H)
    Wb = synth.dense_input(synth.DenseShape(M=1, I=I + offset, H=H), seed=5)[1]
    Wd = Wb.reshape(-1).cuda()[offset:offset + H * I].reshape(H, I)
    W = Wb.reshape(-1)[offset:offset + H * I].reshape(H, I).contiguous()
    Xs, Xd = [], []
    for k, M in enumerate(Ms):
        Xb = synth.dense_input(synth.DenseShape(M=M, I=I + offset, H=1), seed=40 + k)[0]
        Xs.append(Xb.reshape(-1)[offset:offset + M * I].reshape(M, I).contiguous())
        Xd.append(Xb.reshape(-1).cuda()[offset:offset + M * I].reshape(M, I))
    Yg = [poisoned((M, H)) for M in Ms]
    plan = csa.DenseGroupedPlan(Yg, Xd, Wd, I, H)
    assert plan._ws is not None
    for _ in range(2):
        plan()
    Ys = [poisoned((M, H)) for M in Ms]
    for Y, X in zip(Ys, Xd):
        csa.dense_xwt(Y, X, Wd, X.shape[0], I, H)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    wbits = synth.bf16_bits(W).reshape(-1)
    for g, (a, b, X) in enumerate(zip(Yg, Ys, Xs)):
        assert np.array_equal(f32_bits(a), f32_bits(b)), f"problem {g}"
        M = X.shape[0]
        rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, size=4)]))
        ref = oracle_lib.dense_rows(synth.bf16_bits(X).reshape(-1), wbits, M, I, H, rows)
        assert_close(a[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, f"problem {g}")


def test_dense_grouped_realigned_more_than_one_launch():
    """50 problems with I = 770: two copy + grouped launches (48 + 2), W copied once."""
    I, H = 770, 136
    Ms = [16 * (1 + (7 * k) % 23) for k in range(50)]
    W = synth.dense_input(synth.DenseShape(M=1, I=I, H=H), seed=9)[1].cuda()
    Xd = [synth.dense_input(synth.DenseShape(M=M, I=I, H=1), seed=200 + k)[0].cuda()
          for k, M in enumerate(Ms)]
    Yg = [poisoned((M, H)) for M in Ms]
    csa.dense_xwt_grouped(Yg, Xd, W, I, H)
    Ys = [poisoned((M, H)) for M in Ms]
    for Y, X in zip(Ys, Xd):
        csa.dense_xwt(Y, X, W, X.shape[0], I, H)
    torch.cuda.synchronize()
    assert csa.get_status() == 0
    for g, (a, b) in enumerate(zip(Yg, Ys)):
        assert np.array_equal(f32_bits(a), f32_bits(b)), f"problem {g}"
