"""The C ABI on the CPU: the library loads, exports every symbol include/csa.h
declares, and rejects invalid arguments before touching a device."""
import ctypes
import os
import re

import pytest

from causal_attention_score_gb300 import _lib, build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return _lib.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "csa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"trimul_forward", "trimul_forward_ex", "dense_xwt", "dense_xwt_ex",
            "csa_get_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in csa.h but not exported"
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature in the binding"


def test_checking_build_compiles_and_exports_every_symbol():
    """The -DCSA_DEBUG variant (device-side index checks) builds from the same
    sources and exports the same C ABI."""
    path = build_lib.build(debug=True)
    dbg = ctypes.CDLL(path)
    for n in _declared_functions():
        assert hasattr(dbg, n), f"{n} missing from the checking build"
    dbg.csa_status_string.restype = ctypes.c_char_p
    assert b"check" in dbg.csa_status_string(_lib.CSA_ERR_CHECK)


def test_status_strings(lib):
    for code in range(-11, 1):
        assert lib.csa_status_string(code)
        assert lib.csa_status_string(code) != b"unknown status"
    assert lib.csa_version().decode().endswith("sm_103a")


@pytest.mark.parametrize("args,code", [
    ((None, 16, 1, 1, 8, 1), _lib.CSA_ERR_NULL),
    ((16, None, 1, 1, 8, 1), _lib.CSA_ERR_NULL),
    ((16, 16, 0, 1, 8, 1), _lib.CSA_ERR_SHAPE),
    ((16, 16, 1, 0, 8, 1), _lib.CSA_ERR_SHAPE),
    ((16, 16, 1, 1, 10, 3), _lib.CSA_ERR_SHAPE),       # C % NH != 0
    ((16, 16, 1, 1, 12, 1), _lib.CSA_ERR_ALIGN),       # HS = 12
    ((16, 16, 1, 1, 512, 1), _lib.CSA_ERR_UNSUPPORTED),  # HS = 512
    ((16, 8, 1, 1, 64, 1), _lib.CSA_ERR_ALIGN),        # qkv not 16-byte aligned
    ((18, 16, 1, 1, 64, 1), _lib.CSA_ERR_ALIGN),       # out not 4-byte aligned
])
def test_trimul_argument_errors(lib, args, code):
    assert lib.trimul_forward(*args) == code
    assert lib.csa_last_error()


def test_trimul_unknown_flags(lib):
    assert lib.trimul_forward_ex(16, 16, 1, 1, 64, 1, 0, 8, None) == _lib.CSA_ERR_UNSUPPORTED


@pytest.mark.parametrize("args,code", [
    ((None, 16, 16, 1, 1, 1), _lib.CSA_ERR_NULL),
    ((16, 16, 16, 0, 1, 1), _lib.CSA_ERR_SHAPE),
    ((16, 16, 16, 1, -1, 1), _lib.CSA_ERR_SHAPE),
    ((16, 17, 16, 1, 1, 1), _lib.CSA_ERR_ALIGN),
    ((18, 16, 16, 1, 1, 1), _lib.CSA_ERR_ALIGN),
])
def test_dense_argument_errors(lib, args, code):
    assert lib.dense_xwt(*args) == code


def test_no_device_is_an_error_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert lib.trimul_forward(1024, 1024, 1, 64, 128, 2) == _lib.CSA_ERR_CUDA
    assert lib.dense_xwt(1024, 1024, 1024, 4, 4, 4) == _lib.CSA_ERR_CUDA
    assert lib.csa_get_status(None) == _lib.CSA_ERR_CUDA


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import causal_attention_score_gb300 as csa
    qkv = torch.zeros((1, 4, 3, 1, 8), dtype=torch.bfloat16)
    out = torch.zeros((1, 1, 4, 4))
    with pytest.raises(ValueError):
        csa.trimul_forward(out, qkv, 1, 4, 8, 1)


def test_grouped_plan_checks_its_arguments_on_the_host(lib):
    """DenseGroupedPlan refuses bad arguments before anything reaches the library:
    unequal or empty lists, a wrong row length, CPU tensors."""
    import torch
    import causal_attention_score_gb300 as csa
    W = torch.zeros((8, 16), dtype=torch.bfloat16)
    X = torch.zeros((3, 16), dtype=torch.bfloat16)
    Y = torch.zeros((3, 8))
    with pytest.raises(ValueError):
        csa.DenseGroupedPlan([Y, Y], [X], W, 16, 8)
    with pytest.raises(ValueError):
        csa.DenseGroupedPlan([], [], W, 16, 8)
    with pytest.raises(ValueError):
        csa.DenseGroupedPlan([Y], [torch.zeros((3, 15), dtype=torch.bfloat16)], W, 16, 8)
    with pytest.raises(ValueError):  # W (and X, Y) on the CPU
        csa.DenseGroupedPlan([Y], [X], W, 16, 8)
    with pytest.raises(ValueError):
        csa.dense_xwt_grouped([Y], [X], W, 16, 8)


@pytest.mark.parametrize("args,code", [
    ((None, 16, 1, 1, 8, 1, 0, 0, None), _lib.CSA_ERR_NULL),
    ((16, 16, 1, 1, 10, 3, 0, 0, None), _lib.CSA_ERR_SHAPE),
    ((16, 16, 1, 1, 12, 1, 0, 0, None), _lib.CSA_ERR_ALIGN),
    ((16, 16, 1, 1, 64, 1, 0, 4, None), _lib.CSA_ERR_UNSUPPORTED),
])
def test_noalloc_argument_errors(lib, args, code):
    assert lib.trimul_forward_noalloc(*args) == code


@pytest.mark.parametrize("args,code", [
    ((None, 16, 1, 1, 8, 1, 0, 0, None), _lib.CSA_ERR_NULL),
    ((16, None, 1, 1, 8, 1, 0, 0, None), _lib.CSA_ERR_NULL),
    ((16, 16, 0, 1, 8, 1, 0, 0, None), _lib.CSA_ERR_SHAPE),
    ((16, 16, 1, 1, 10, 3, 0, 0, None), _lib.CSA_ERR_SHAPE),      # C % NH != 0
    ((16, 16, 1, 1, 6, 1, 0, 0, None), _lib.CSA_ERR_ALIGN),       # HS = 6 (fp32 needs HS % 4)
    ((16, 16, 1, 1, 260, 1, 0, 0, None), _lib.CSA_ERR_UNSUPPORTED),  # HS = 260
    ((16, 8, 1, 1, 64, 1, 0, 0, None), _lib.CSA_ERR_ALIGN),       # qkv not 16-byte aligned
    ((18, 16, 1, 1, 64, 1, 0, 0, None), _lib.CSA_ERR_ALIGN),      # out not 4-byte aligned
    ((16, 16, 1, 1, 64, 1, 0, 2, None), _lib.CSA_ERR_UNSUPPORTED),  # unknown flag
])
def test_trimul_f32_argument_errors(lib, args, code):
    assert lib.trimul_forward_f32(*args) == code
    assert lib.csa_last_error()


@pytest.mark.parametrize("args,code", [
    ((None, 16, 1, 1, 8, 1, None), _lib.CSA_ERR_NULL),
    ((16, None, 1, 1, 8, 1, None), _lib.CSA_ERR_NULL),
    ((16, 16, 1, 0, 8, 1, None), _lib.CSA_ERR_SHAPE),
    ((16, 16, 1, 1, 10, 3, None), _lib.CSA_ERR_SHAPE),
    ((16, 16, 1, 1, 12, 1, None), _lib.CSA_ERR_ALIGN),             # HS = 12
    ((16, 16, 1, 1, 256, 1, None), _lib.CSA_ERR_UNSUPPORTED),      # HS = 256 (softmax: <= 128)
    ((16, 8, 1, 1, 64, 1, None), _lib.CSA_ERR_ALIGN),
])
def test_softmax_argument_errors(lib, args, code):
    assert lib.causal_softmax_forward(*args) == code
    assert lib.csa_last_error()


@pytest.mark.parametrize("args,code", [
    ((None, 16, 16, 1, 1, 1, 8, None), _lib.CSA_ERR_NULL),
    ((16, 16, 16, 0, 1, 1, 8, None), _lib.CSA_ERR_SHAPE),
    ((16, 16, 16, 1, 1, 1, 12, None), _lib.CSA_ERR_ALIGN),         # D = 12
    ((16, 16, 16, 1, 1, 1, 264, None), _lib.CSA_ERR_UNSUPPORTED),  # D = 264
    ((16, 8, 16, 1, 1, 1, 64, None), _lib.CSA_ERR_ALIGN),          # X not 16-byte aligned
])
def test_bmm_nt_argument_errors(lib, args, code):
    assert lib.batch_matmul_nt(*args) == code


def test_no_device_for_the_other_entry_points(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert lib.trimul_forward_f32(1024, 1024, 1, 64, 128, 2, 0, 0, None) == _lib.CSA_ERR_CUDA
    assert lib.causal_softmax_forward(1024, 1024, 1, 64, 128, 2, None) == _lib.CSA_ERR_CUDA
    assert lib.batch_matmul_nt(1024, 1024, 1024, 2, 8, 8, 64, None) == _lib.CSA_ERR_CUDA


def _grouped_args(ys, xs, ms):
    n = len(ms)
    y = (ctypes.c_void_p * n)(*ys)
    x = (ctypes.c_void_p * n)(*xs)
    m = (ctypes.c_int * n)(*ms)
    return y, x, m


@pytest.mark.parametrize("ys,xs,ms,n,code", [
    ([1024, 2048], [1024, 2048], [4, 4], 0, _lib.CSA_ERR_SHAPE),        # n = 0
    ([1024, None], [1024, 2048], [4, 4], 2, _lib.CSA_ERR_NULL),         # Y[1] null
    ([1024, 2048], [None, 2048], [4, 4], 2, _lib.CSA_ERR_NULL),         # X[0] null
    ([1024, 2048], [1024, 2048], [4, 0], 2, _lib.CSA_ERR_SHAPE),        # M[1] = 0
    ([1024, 2050], [1024, 2048], [4, 4], 2, _lib.CSA_ERR_ALIGN),        # Y[1] 2-byte aligned
    ([1024, 2048], [1024, 2049], [4, 4], 2, _lib.CSA_ERR_ALIGN),        # X[1] odd address
])
def test_dense_grouped_argument_errors(lib, ys, xs, ms, n, code):
    y, x, m = _grouped_args(ys, xs, ms)
    rc = lib.dense_xwt_grouped(ctypes.addressof(y), ctypes.addressof(x), 4096,
                               ctypes.addressof(m), n, 8, 8, None)
    assert rc == code
    assert lib.csa_last_error()


def test_dense_grouped_null_arrays_and_no_device(lib):
    y, x, m = _grouped_args([1024], [2048], [4])
    assert lib.dense_xwt_grouped(None, ctypes.addressof(x), 4096, ctypes.addressof(m), 1, 8, 8,
                                 None) == _lib.CSA_ERR_NULL
    assert lib.dense_xwt_grouped(ctypes.addressof(y), ctypes.addressof(x), 4096, None, 1, 8, 8,
                                 None) == _lib.CSA_ERR_NULL
    assert lib.dense_xwt_grouped(ctypes.addressof(y), ctypes.addressof(x), 4097,
                                 ctypes.addressof(m), 1, 8, 8, None) == _lib.CSA_ERR_ALIGN
    import torch
    if torch.cuda.is_available():
        return
    assert lib.dense_xwt_grouped(ctypes.addressof(y), ctypes.addressof(x), 4096,
                                 ctypes.addressof(m), 1, 8, 8, None) == _lib.CSA_ERR_CUDA


def test_wait_limit_default_setter_and_environment(lib):
    """The watchdog bound: 2 s by default, set and restored through the API, and taken
    from CSA_WAIT_LIMIT_NS when that holds a positive integer (a fresh process)."""
    import subprocess
    import sys
    assert lib.csa_get_wait_limit_ns() == 2_000_000_000 or os.environ.get("CSA_WAIT_LIMIT_NS")
    lib.csa_set_wait_limit_ns(12345)
    assert lib.csa_get_wait_limit_ns() == 12345
    lib.csa_set_wait_limit_ns(0)
    code = ("import causal_attention_score_gb300 as c; print(c.get_wait_limit_ns())")
    for env, want in (("50000000", 50_000_000), ("junk", 2_000_000_000), ("0", 2_000_000_000)):
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True,
                             text=True, env={**os.environ, "CSA_WAIT_LIMIT_NS": env}, check=True)
        assert int(out.stdout.strip()) == want, (env, out.stdout, out.stderr)


def _ws_bytes(lib, X, W, M, I, H):
    n = ctypes.c_size_t(123)
    rc = lib.dense_xwt_workspace_size(X, W, M, I, H, ctypes.byref(n))
    return rc, n.value


def test_dense_workspace_size(lib):
    """No workspace when tensor maps describe the rows as they are; otherwise the
    realigned copy (rows padded to 64 elements, X's part 256-byte rounded) and 256
    bytes of alignment slack."""
    P = (770 + 63) // 64 * 64
    r256 = lambda n: (n + 255) // 256 * 256
    assert _ws_bytes(lib, 4096, 8192, 960, 768, 768) == (0, 0)
    assert _ws_bytes(lib, 4096, 8192, 960, 770, 768) == (
        0, 256 + r256(960 * P * 2) + 768 * P * 2)
    # a misaligned view needs the copy even when I * 2 is a multiple of 16
    rc, n = _ws_bytes(lib, 4098, 8192, 10, 768, 20)
    assert rc == 0 and n == 256 + r256(10 * 768 * 2) + 20 * 768 * 2  # 768 is a multiple of 64
    assert _ws_bytes(lib, None, 8192, 1, 1, 1)[0] == _lib.CSA_ERR_NULL
    assert _ws_bytes(lib, 16, 16, 0, 1, 1) == (_lib.CSA_ERR_SHAPE, 0)
    assert lib.dense_xwt_workspace_size(16, 16, 1, 1, 1, None) == _lib.CSA_ERR_NULL


def test_dense_ws_rejects_missing_small_or_misaligned_workspace(lib):
    """Checked before any device is touched (this host has none)."""
    _, need = _ws_bytes(lib, 4096, 8192, 960, 770, 768)
    args = (1 << 20, 4096, 8192, 960, 770, 768)
    assert lib.dense_xwt_ws(*args, None, 0, None) == _lib.CSA_ERR_WORKSPACE
    assert b"needed" in lib.csa_last_error()
    assert lib.dense_xwt_ws(*args, 1 << 24, need - 1, None) == _lib.CSA_ERR_WORKSPACE
    assert lib.dense_xwt_ws(*args, (1 << 24) + 8, need, None) == _lib.CSA_ERR_ALIGN
    assert lib.dense_xwt_ws(None, 4096, 8192, 960, 770, 768, 1 << 24, need,
                            None) == _lib.CSA_ERR_NULL


def test_library_sources_call_no_device_allocator():
    """Every device buffer belongs to the caller: no source of the library calls a
    device allocator or a memory pool (its only device memory is fixed arrays)."""
    csrc = os.path.join(ROOT, "causal_attention_score_gb300", "csrc")
    pat = re.compile(r"cuda(Malloc|Free)(?!Host)|cudaMemPool|cuMem(Alloc|Create|Free)")
    for f in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, f), encoding="utf-8").read()
        code = re.sub(r"//[^\n]*", "", re.sub(r"/\*.*?\*/", "", text, flags=re.S))
        assert not pat.search(code), f"{f} calls a device allocator"


def test_library_is_stamped_with_its_sources(tmp_path, monkeypatch):
    """build() stamps the library with a hash of its sources; a source edit makes the
    stamp stale (so build() rebuilds and the binding refuses the old binary)."""
    path = build_lib.build()
    assert build_lib.up_to_date(path)
    with open(build_lib.stamp_path(path)) as f:
        assert f.read().strip() == build_lib.source_hash()
    extra = tmp_path / "extra.h"
    extra.write_text("// one more header\n")
    deps = build_lib._deps()
    monkeypatch.setattr(build_lib, "_deps", lambda: deps + [str(extra)])
    assert not build_lib.up_to_date(path)
    assert build_lib.source_hash() != build_lib.source_hash(debug=True)


def test_dense_grouped_workspace_size_and_errors(lib):
    P = (770 + 63) // 64 * 64
    r256 = lambda n: (n + 255) // 256 * 256
    n = ctypes.c_size_t(5)
    xs = (ctypes.c_void_p * 3)(4096, 8192, 16384)
    ms = (ctypes.c_int * 3)(10, 300, 1)
    ys = (ctypes.c_void_p * 3)(1 << 20, 1 << 21, 1 << 22)
    assert lib.dense_xwt_grouped_workspace_size(xs, 4096, ms, 3, 768, 64, ctypes.byref(n)) == 0
    assert n.value == 0
    assert lib.dense_xwt_grouped_workspace_size(xs, 4096, ms, 3, 770, 64, ctypes.byref(n)) == 0
    assert n.value == 256 + r256(64 * P * 2) + sum(r256(m * P * 2) for m in (10, 300, 1))
    assert lib.dense_xwt_grouped_workspace_size(xs, 4096, ms, 0, 770, 64, ctypes.byref(n)) == \
        _lib.CSA_ERR_SHAPE
    assert lib.dense_xwt_grouped_ws(ys, xs, 4096, ms, 3, 770, 64, 1 << 24, 10, None) == \
        _lib.CSA_ERR_WORKSPACE
    need = 256 + r256(64 * P * 2) + sum(r256(m * P * 2) for m in (10, 300, 1))
    assert lib.dense_xwt_grouped_ws(ys, xs, 4096, ms, 3, 770, 64, (1 << 24) + 8, need, None) == \
        _lib.CSA_ERR_ALIGN


def test_stream_sm_limits_on_the_host(lib):
    """Per-stream SM limits are host state: set, read back, replaced, removed; a
    negative limit is refused; at most 64 streams carry one (then CSA_ERR_BUSY)."""
    v = ctypes.c_int(-1)
    s1, s2 = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000)
    assert lib.csa_get_stream_sm_limit(s1, ctypes.byref(v)) == 0 and v.value == 0
    assert lib.csa_set_stream_sm_limit(s1, 100) == 0
    assert lib.csa_set_stream_sm_limit(s2, 52) == 0
    assert lib.csa_get_stream_sm_limit(s1, ctypes.byref(v)) == 0 and v.value == 100
    assert lib.csa_get_stream_sm_limit(s2, ctypes.byref(v)) == 0 and v.value == 52
    assert lib.csa_set_stream_sm_limit(s1, 96) == 0
    assert lib.csa_get_stream_sm_limit(s1, ctypes.byref(v)) == 0 and v.value == 96
    assert lib.csa_set_stream_sm_limit(s1, -1) == _lib.CSA_ERR_SHAPE
    assert lib.csa_get_stream_sm_limit(s1, ctypes.byref(v)) == 0 and v.value == 96
    assert lib.csa_get_stream_sm_limit(s1, None) == _lib.CSA_ERR_NULL
    for s in (s1, s2):
        assert lib.csa_set_stream_sm_limit(s, 0) == 0
        assert lib.csa_get_stream_sm_limit(s, ctypes.byref(v)) == 0 and v.value == 0
    assert lib.csa_set_stream_sm_limit(s1, 0) == 0  # removing an absent limit is fine
    handles = [ctypes.c_void_p(0x10000 + 16 * i) for i in range(65)]
    try:
        for h in handles[:64]:
            assert lib.csa_set_stream_sm_limit(h, 8) == 0
        assert lib.csa_set_stream_sm_limit(handles[64], 8) == _lib.CSA_ERR_BUSY
        assert lib.csa_set_stream_sm_limit(handles[3], 0) == 0
        assert lib.csa_set_stream_sm_limit(handles[64], 8) == 0
        assert lib.csa_get_stream_sm_limit(handles[63], ctypes.byref(v)) == 0 and v.value == 8
    finally:
        for h in handles:
            lib.csa_set_stream_sm_limit(h, 0)


def test_dense_tiling_rule(lib):
    """The single-call tiling on a 152-SM GB300, worked by hand from the cost model
    (waves of 128 x BN units over the SMs, or of 256 x BN pair units over 76 clusters,
    each wave costing BN + 32; pairs on a strictly lower cost, or an equal one with at
    least three pair tiles per cluster)."""
    bn, pairs = ctypes.c_int(0), ctypes.c_int(0)

    def tiling(M, H, sms):
        assert lib.csa_dense_tiling(M, H, sms, ctypes.byref(bn), ctypes.byref(pairs)) == 0
        return bn.value, pairs.value

    # M = 1088: 9 m-tiles. Single: BN 192 -> 144 tiles, one wave, cost 224 (BN 256: 288).
    # Pairs: 5 rows; BN 256 -> 60 tiles, one wave, 288; BN 192 -> 80 > 76, two waves.
    assert tiling(1088, 3072, 152) == (192, 0)
    # M = 6144: 48 m-tiles. Single: BN 256 -> 576 tiles, 4 waves, 1152 (192: 6 x 224 =
    # 1344; 128: 8 x 160 = 1280). Pairs: 24 rows, BN 256 -> 288 tiles, 4 waves, 1152:
    # equal, and 288 >= 3 x 76.
    assert tiling(6144, 3072, 152) == (256, 1)
    # M = 4096: single BN 256, 384 tiles, 3 waves, 864; pairs BN 256, 192 tiles, 3 waves,
    # 864: equal, but 192 < 228 pair tiles.
    assert tiling(4096, 3072, 152) == (256, 0)
    # One SM leaves no cluster of two.
    assert tiling(32768, 3072, 1)[1] == 0
    assert tiling(32768, 3072, 152)[1] == 1
    assert lib.csa_dense_tiling(0, 3072, 152, ctypes.byref(bn), ctypes.byref(pairs)) == \
        _lib.CSA_ERR_SHAPE
    assert lib.csa_dense_tiling(64, 64, 0, ctypes.byref(bn), ctypes.byref(pairs)) == \
        _lib.CSA_ERR_SHAPE
    assert lib.csa_dense_tiling(64, 64, 152, None, ctypes.byref(pairs)) == _lib.CSA_ERR_NULL
