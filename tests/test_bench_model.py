"""The benchmark's work and traffic model against the numbers the pages print (CPU)."""
import os

import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


def test_tiled_traffic_matches_kernl_worked_example():
    for M, N, K, bM, bN, bK, loads, writes in _rows("kernl_tiled_matmul_traffic.txt"):
        got = bench.tiled_traffic(int(M), int(N), int(K), int(bM), int(bN), int(bK))
        assert got == (int(loads), int(writes))


def test_smaller_tiles_load_more():
    # the tutorial's closing remark: smaller block_M / block_N increase the loads
    base = bench.tiled_traffic(15, 9, 12, 5, 3, 6)[0]
    assert bench.tiled_traffic(15, 9, 12, 3, 3, 6)[0] > base
    assert bench.tiled_traffic(15, 9, 12, 5, 1, 6)[0] > base


def test_dense_flops_and_raggedness_of_dietcode_workload():
    (name, B, T, I, H, _), = [r for r in _rows("dietcode_workloads.txt") if r[0] == "dense"]
    B, T, I, H = int(B), int(T), int(I), int(H)
    assert bench.dense_flops(B * T, I, H) == 2 * 16 * 60 * 770 * 2304
    assert (B * T) % 128 != 0 and I % 4 != 0 and B * T == 960


def test_trimul_flops_counts_lower_triangle_including_diagonal():
    # T=1: one score per head; T=2: three; a full T x T product would give T^2
    assert bench.trimul_flops(1, 1, 64, 1) == 2 * 64
    assert bench.trimul_flops(1, 2, 64, 1) == 3 * 2 * 64
    assert bench.trimul_flops(8, 1024, 768, 12) == 6_448_742_400


def test_algorithmic_bytes():
    assert bench.trimul_algorithmic_bytes(8, 1024, 768, 12) == 8 * 12 * 1024 * 1024 * 4 + 2 * 8 * 1024 * 768 * 2
    assert bench.trimul_algorithmic_bytes(1, 4, 8, 1, lower_only=True) == 10 * 4 + 2 * 4 * 8 * 2
    assert bench.dense_algorithmic_bytes(960, 770, 768) == (960 + 768) * 770 * 2 + 960 * 768 * 4


def test_traffic_record_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    """roofline.traffic is taken from a committed ncu record only while the score
    kernel's code is the one it was captured on: a comment edit keeps it, a code
    edit drops it."""
    src = tmp_path / "k.cu"
    src.write_text("// a kernel\n__global__ void k(int* p) { p[0] = 1; }  /* tail */\n")
    monkeypatch.setattr(bench, "KERNEL_SOURCES", [str(src)])
    h0 = bench.kernel_source_hash()
    src.write_text("// a kernel, described at length\n/* block\n comment */\n"
                   "__global__ void k(int* p) {\n  p[0] = 1;  // store\n}\n")
    assert bench.kernel_source_hash() == h0
    src.write_text("// a kernel\n__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench.kernel_source_hash() != h0



def test_step_time_percentiles_match_numpy():
    import numpy as np
    rng = np.random.default_rng(1)
    for n in (1, 2, 7, 200):
        xs = rng.uniform(0.05, 0.09, size=n).tolist()
        for q in (10, 50, 90):
            assert abs(bench._percentile(xs, q) - float(np.percentile(xs, q))) < 1e-12


def test_oracle_samples_cover_one_step():
    """The default step's CPU baseline samples are 1/32 of a step each: 32 consecutive
    samples compute every head of the long-context scores once and every row of the 33
    dense problems once, i.e. exactly one step's useful flops."""
    from causal_attention_score_gb300 import synth
    sample = bench.OracleSample("step")
    tl = synth.TRIMUL_LONG
    xs, W = synth.dense_sweep_inputs(seed=0)
    H, I = W.shape
    step = (bench.trimul_flops(tl.B, tl.T, tl.C, tl.NH)
            + sum(bench.dense_flops(X.shape[0], I, H) for X in xs)
            + bench.dense_flops(synth.DENSE_RAGGED.M, synth.DENSE_RAGGED.I, synth.DENSE_RAGGED.H))
    assert step == 226_755_411_968
    assert sum(sample.flops(i) for i in range(32)) == step
    heads = {tuple(sample.parts(i)[0][0, :2]) for i in range(32)}
    assert len(heads) == tl.B * tl.NH
