"""Benchmark of the hot path. One step is one pass over every stage of the path on the
largest configurations the pages give:

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--graph]

Default step (workload "step"; seeded synthetic data, resident in HBM before timing):
  trimul_forward     the causal scores of QKV bf16 (B=2, T=4096, 3, NH=16, HS=128), N(0,1)
                     seed 0 -> fp32 (2, 16, 4096, 4096), NaN above the diagonal (the long
                     context; the score product of "llm.c dev/cuda/trimat_forward.cu");
  dense_xwt_grouped  the dynamic-shape sweep: 32 problems X_i [16*T_i, 768], T_i ~ U{1..128}
                     (seed 0), X_i uniform[-1,1] (seed 1000+i), sharing W [3072, 768]
                     (uniform[-1,1], seed 1), in one launch;
  dense_xwt          the ragged layer X [960, 770], W [768, 770], uniform[-1,1] seed 0
                     (B*T = 16*60 and I = 770 of "DietCode ... test_local_padding").
Metric: useful TFLOP/s = (lower-triangle flops 2*HS*B*NH*T(T+1)/2 + dense flops 2*M*I*H)
per step / step time. L2 is flushed (256 MiB write) between timed steps, outside the timed
events; the timed region has one event before and one after each step. Before it, the step
runs back to back for a clock soak (--soak-ms) so that the timed steps see steady clocks;
NVML clock samples are taken through the soak and the timed region. Per-part times (and
each kernel's launch duration, the `rooflines` entries) come from a second pass of the same
K steps with an event after each part; the sweep's 32 problems are also timed as 32
separate dense_xwt calls in a third pass (`sweep_calls`). Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle (the only other implementation of the
method; the pages ship no runnable GPU code) on the host cores, each step a bounded
sample (1/32) of the same workload, and prints the same line.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "useful TFLOP/s (lower-triangle FLOPs) and % of GB300 bf16 dense peak"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 * 1024 * 1024
# The default step runs its dense calls on a stream limited to this many SMs,
# launched first, beside the score kernel on a stream of its own: the score kernel
# starts on the other SMs and takes the rest as the dense kernels finish (its work
# list is dynamic). Measured over limits 32-80 on a GB300 (L2 flushed): 56 best,
# 439 us per step against 467 us with the three calls one after another.
STEP_DENSE_SMS = 56


# --------------------------------------------------------------- work model --

def trimul_flops(B, T, C, NH):
    """Useful flops of the causal product: 2*HS per score, lower triangle incl. diagonal."""
    HS = C // NH
    return 2 * HS * B * NH * T * (T + 1) // 2


def dense_flops(M, I, H):
    """2*M*I*H, the count "DietCode ... test_local_padding" divides by time."""
    return 2 * M * I * H


def dense_algorithmic_bytes(M, I, H):
    """X and W read once (bf16), Y written once (fp32)."""
    return (M * I + H * I) * 2 + M * H * 4


def trimul_algorithmic_bytes(B, T, C, NH, lower_only=False, in_bytes=2):
    """Minimum HBM traffic of one trimul_forward: every output element written once
    (fp32), Q and K read once (bf16, or fp32 with in_bytes=4); V is never touched."""
    out = B * NH * (T * (T + 1) // 2 if lower_only else T * T) * 4
    qk = 2 * B * T * C * in_bytes
    return out + qk


def dense_algorithmic_bytes(M, I, H):
    return (M * I + H * I) * 2 + M * H * 4


def tiled_traffic(M, N, K, bM, bN, bK):
    """Global-memory element loads and writes of a tiled matmul that fetches an
    A tile and a B tile per (M, N, K) tile step and writes each output tile once
    ("kernl tutorial 1 - tiled matmul": loads (bM*bK + bK*bN) * K/bK * N/bN * M/bM,
    writes M*N)."""
    steps = math.ceil(M / bM) * math.ceil(N / bN) * math.ceil(K / bK)
    return (bM * bK + bK * bN) * steps, M * N


# ---------------------------------------------------------- distributed --

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("CSA_BENCH_BACKEND", "nccl")
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (the job's elapsed time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks --

_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
            0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
            0x80: "hw_power_brake_slowdown", 0x100: "display_clocks"}


class ClockSampler:
    """Reads SM clock and clock-event reasons through NVML (read-only) in a thread."""

    def __init__(self, index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._ok = False
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index),
                                                       ctypes.byref(self.handle)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self._reasons_fn = fn
            self._ok = True
        except OSError:
            self._ok = False

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0:
                self.samples.append(int(clk.value))
            if self._reasons_fn(self.handle, ctypes.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(self.period)

    def start(self):
        if self._ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread:
            self._stop.set()
            self._thread.join()

    def summary(self):
        if not self._ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        names = [n for bit, n in _REASONS.items() if self.reasons & bit]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples)}


def nvml_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p for p in vis.split(",") if p.strip()]
    if parts and parts[min(local_rank, len(parts) - 1)].strip().isdigit():
        return int(parts[min(local_rank, len(parts) - 1)])
    return local_rank


CSRC = os.path.join(ROOT, "causal_attention_score_gb300", "csrc")
KERNEL_SOURCES = [os.path.join(CSRC, f) for f in ("trimul_sm103a.cu", "sm103a_ptx.cuh")]
DENSE_SOURCES = [os.path.join(CSRC, f) for f in ("dense_sm103a.cu", "sm103a_ptx.cuh")]
# Committed ncu records of DRAM bytes per launch: record name -> (file, kernel sources).
TRAFFIC_RECORDS = {
    "trimul_long": ("trimul_long_dram_traffic.txt", "KERNEL_SOURCES"),
    "trimul_gpt2": ("trimul_gpt2_dram_traffic.txt", "KERNEL_SOURCES"),
    "dense_sweep_grouped": ("dense_sweep_grouped_dram_traffic.txt", "DENSE_SOURCES"),
    "dense_ragged": ("dense_ragged_dram_traffic.txt", "DENSE_SOURCES"),
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "trimul_gpt2_dram_traffic.txt")


def kernel_source_hash(sources=None) -> str:
    """Hash of a kernel's code with comments and blank space removed, so that an edit
    of its comments keeps a traffic record taken on the same code."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in (KERNEL_SOURCES if sources is None else sources):
        with open(f, encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)  # block comments
        src = re.sub(r"//[^\n]*", " ", src)                # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(record: str = "trimul_gpt2"):
    """DRAM bytes (read + write) per launch from a committed ncu summary, or None when
    there is none or the kernel's code changed since it was taken."""
    fname, sources = TRAFFIC_RECORDS[record]
    path = TRAFFIC_FILE if record == "trimul_gpt2" else os.path.join(ROOT, "profiles", fname)
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != kernel_source_hash(globals()[sources]):
            return None
        return float(kv["dram_bytes_per_launch_full_size"])
    except (OSError, KeyError, ValueError):
        return None


def _percentile(xs, q):
    """q-th percentile (linear interpolation) of a non-empty list."""
    v = sorted(xs)
    pos = (len(v) - 1) * q / 100.0
    lo = int(math.floor(pos))
    hi = min(lo + 1, len(v) - 1)
    return v[lo] + (v[hi] - v[lo]) * (pos - lo)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------ our arm --

class Part:
    """One launch (or call) of a step: a label, fn(stream), the number of this
    library's kernels it launches, and its roofline terms: kernel name, bound
    ("hbm" or "tensor"), algorithmic bytes or flops per launch, and the name of
    the committed DRAM traffic record, if any."""

    def __init__(self, label, fn, kernels=1, kernel=None, bound=None, per_launch=None,
                 traffic=None, hbm_bytes=None):
        self.label = label
        self.hbm_bytes = hbm_bytes  # algorithmic HBM bytes of one launch (all parts)
        self.fn = fn
        self.kernels = kernels
        self.kernel = kernel
        self.bound = bound
        self.per_launch = per_launch
        self.traffic = traffic


class Workload:
    """What one step runs: parts timed back to back with CUDA events, the useful flops
    of a step, the host<->device copies of the end-to-end variant, optional separate
    calls timed one by one (`calls`: [(label, M, flops, fn)]) and the oracle sample
    that stands for a bounded part of the step on the CPU."""

    def __init__(self, name, config, parts, flops, h2d, d2h, dtype="bf16",
                 data="synthetic (seeded N(0,1) / uniform[-1,1], rounded to bf16)", calls=None,
                 branches=None):
        self.name = name          # human-readable workload string (config.workload)
        self.dtype = dtype        # arithmetic type of the path
        self.data = data
        self.config = config      # extra config keys
        self.parts = parts        # [Part]
        self.flops = flops        # useful flops per step
        self.h2d = h2d            # [(device tensor, host tensor)]
        self.d2h = d2h            # [(host tensor, device tensor)]
        self.calls = calls or []
        # Concurrent schedule of a timed step: [(sm_limit, [Part])], each branch on a
        # stream of its own (0: no SM limit), launched in this order after a fork from
        # the step's stream and joined back into it; None: the parts one after another.
        self.branches = branches
        self.kernels_per_step = sum(p.kernels for p in parts)


def make_workload(name, dev):
    import torch

    import causal_attention_score_gb300 as csa
    from causal_attention_score_gb300 import synth

    def trimul_part(shape, lower_only=False, seed=0, traffic=None):
        qkv_h = synth.trimul_input(shape, seed=seed, dist="normal")
        qkv = qkv_h.to(dev)
        out = torch.empty(shape.out_shape, dtype=torch.float32, device=dev)
        fn = lambda st: csa.trimul_forward(out, qkv, shape.B, shape.T, shape.C, shape.NH,
                                           lower_only=lower_only, stream=st)
        nbytes = trimul_algorithmic_bytes(shape.B, shape.T, shape.C, shape.NH, lower_only)
        part = Part("trimul", fn, kernel="trimul_sm103a_kernel", bound="hbm",
                    per_launch=nbytes, traffic=traffic, hbm_bytes=nbytes)
        return part, [(qkv, qkv_h)], [out]

    def dense_part(shape, seed=0, label="dense_ragged", traffic="dense_ragged"):
        X_h, W_h = synth.dense_input(shape, seed=seed)
        X, W = X_h.to(dev), W_h.to(dev)
        Y = torch.empty((shape.M, shape.H), dtype=torch.float32, device=dev)
        # The workspace the realigning fetch needs (I = 770 rows are not 16-byte
        # multiples), allocated once like the other buffers.
        nbytes = csa.dense_workspace_size(X, W, shape.M, shape.I, shape.H)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
        fn = lambda st: csa.dense_xwt_ws(Y, X, W, shape.M, shape.I, shape.H, ws, stream=st)
        part = Part(label, fn, kernels=2 if nbytes else 1,
                    kernel="realign_rows_kernel + dense_sm103a_kernel" if nbytes else
                    "dense_sm103a_kernel", bound="tensor",
                    per_launch=dense_flops(shape.M, shape.I, shape.H), traffic=traffic,
                    hbm_bytes=dense_algorithmic_bytes(shape.M, shape.I, shape.H))
        return part, [(X, X_h), (W, W_h)], [Y]

    def sweep_parts():
        xs_h, W_h = synth.dense_sweep_inputs(seed=0)
        W = W_h.to(dev)
        H, I = W_h.shape
        Xs = [X_h.to(dev) for X_h in xs_h]
        Ys = [torch.empty((X.shape[0], H), dtype=torch.float32, device=dev) for X in Xs]
        flops = sum(dense_flops(X.shape[0], I, H) for X in Xs)
        plan = csa.DenseGroupedPlan(Ys, Xs, W, I, H)  # tensors checked once
        part = Part("dense_grouped", lambda st: plan(stream=st),
                    kernel="dense_sm103a_kernel<grouped, CTA pairs>", bound="tensor",
                    per_launch=flops, traffic="dense_sweep_grouped",
                    hbm_bytes=H * I * 2 + sum(X.shape[0] * (I * 2 + H * 4) for X in Xs))
        calls = [(f"call{i}_M{X.shape[0]}", int(X.shape[0]), dense_flops(X.shape[0], I, H),
                  (lambda X, Y: lambda st: csa.dense_xwt(Y, X, W, X.shape[0], I, H,
                                                         stream=st))(X, Y))
                 for i, (X, Y) in enumerate(zip(Xs, Ys))]
        return part, [(W, W_h)] + list(zip(Xs, xs_h)), Ys, flops, calls, (I, H, len(Xs))

    def pinned_like(t):
        return torch.empty(t.shape, dtype=t.dtype, pin_memory=True)

    def finish(wl_name, config, parts, flops, h2d, outs, **kw):
        h2d = [(d, h.pin_memory()) for d, h in h2d]
        d2h = [(pinned_like(o), o) for o in outs]
        return Workload(wl_name, config, parts, flops, h2d, d2h, **kw)

    ts, tl, ds = synth.TRIMUL_GPT2, synth.TRIMUL_LONG, synth.DENSE_RAGGED
    if name == "step":
        tp, th, to = trimul_part(tl, traffic="trimul_long")
        gp, gh, go, gflops, calls, (I, H, n) = sweep_parts()
        dp, dh, do = dense_part(ds)
        return finish(
            "trimul long context (B=2,T=4096,C=2048,NH=16,HS=128) + dense dynamic-shape sweep "
            "(32 problems M=16*T, T~U{1..128} seed 0, I=768, H=3072) in one grouped launch + "
            "dense ragged (M=960,I=770,H=768), one call each per step",
            {"trimul": {"B": tl.B, "T": tl.T, "C": tl.C, "NH": tl.NH, "mask": "NaN"},
             "dense_sweep": {"calls": n, "I": I, "H": H, "grouped": True,
                             "M": [c[1] for c in calls]},
             "dense": {"M": ds.M, "I": ds.I, "H": ds.H}},
            [tp, gp, dp],
            trimul_flops(tl.B, tl.T, tl.C, tl.NH) + gflops + dense_flops(ds.M, ds.I, ds.H),
            th + gh + dh, to + go + do, calls=calls,
            branches=[(STEP_DENSE_SMS, [gp, dp]), (0, [tp])])
    if name == "step_gpt2":
        tp, th, to = trimul_part(ts, traffic="trimul_gpt2")
        dp, dh, do = dense_part(ds)
        return finish(
            "trimul GPT-2-small (B=8,T=1024,C=768,NH=12,HS=64) + dense ragged "
            "(M=960,I=770,H=768), one call each per step",
            {"trimul": {"B": ts.B, "T": ts.T, "C": ts.C, "NH": ts.NH, "mask": "NaN"},
             "dense": {"M": ds.M, "I": ds.I, "H": ds.H}},
            [tp, dp],
            trimul_flops(ts.B, ts.T, ts.C, ts.NH) + dense_flops(ds.M, ds.I, ds.H),
            th + dh, to + do)
    if name in ("trimul_gpt2", "trimul_long", "trimul_gpt2_lower", "trimul_long_lower"):
        shape = ts if "gpt2" in name else tl
        lower = name.endswith("_lower")
        tp, th, to = trimul_part(shape, lower_only=lower,
                                 traffic=None if lower else name)
        return finish(
            f"trimul {'GPT-2-small' if 'gpt2' in name else 'long context'} (B={shape.B},"
            f"T={shape.T},C={shape.C},NH={shape.NH},HS={shape.HS})"
            + (", lower triangle only" if lower else ""),
            {"trimul": {"B": shape.B, "T": shape.T, "C": shape.C, "NH": shape.NH,
                        "mask": "untouched" if lower else "NaN"}},
            [tp], trimul_flops(shape.B, shape.T, shape.C, shape.NH), th, to)
    if name in ("trimul_f32_gpt2", "trimul_f32_long"):
        shape = ts if "gpt2" in name else tl
        qkv_h = synth.trimul_input_f32(shape, seed=0, dist="uniform")
        qkv = qkv_h.to(dev)
        out = torch.empty(shape.out_shape, dtype=torch.float32, device=dev)
        fn = lambda st: csa.trimul_forward_f32(out, qkv, shape.B, shape.T, shape.C, shape.NH,
                                               stream=st)
        part = Part("trimul_f32", fn, kernel="trimul_sm103a_kernel<fp32>", bound="hbm",
                    per_launch=trimul_algorithmic_bytes(shape.B, shape.T, shape.C, shape.NH,
                                                        in_bytes=4))
        return finish(
            f"trimul over fp32 inputs (3 x tf32), {'GPT-2-small' if 'gpt2' in name else 'long context'}"
            f" (B={shape.B},T={shape.T},C={shape.C},NH={shape.NH},HS={shape.HS})",
            {"trimul_f32": {"B": shape.B, "T": shape.T, "C": shape.C, "NH": shape.NH,
                            "mask": "NaN"}},
            [part], trimul_flops(shape.B, shape.T, shape.C, shape.NH),
            [(qkv, qkv_h)], [out], dtype="tf32x3",
            data="synthetic (seeded uniform[-1,1] fp32, not rounded)")
    if name in ("softmax_gpt2", "softmax_long"):
        shape = ts if name == "softmax_gpt2" else tl
        qkv_h = synth.trimul_input(shape, seed=0, dist="normal")
        qkv = qkv_h.to(dev)
        att = torch.empty(shape.out_shape, dtype=torch.float32, device=dev)
        fn = lambda st: csa.causal_softmax_forward(att, qkv, shape.B, shape.T, shape.C, shape.NH,
                                                   stream=st)
        part = Part("softmax", fn, kernel="softmax_sm103a_kernel", bound="hbm",
                    per_launch=trimul_algorithmic_bytes(shape.B, shape.T, shape.C, shape.NH))
        return finish(
            f"causal softmax of the scores, {'GPT-2-small' if name == 'softmax_gpt2' else 'long context'}"
            f" (B={shape.B},T={shape.T},C={shape.C},NH={shape.NH},HS={shape.HS})",
            {"softmax": {"B": shape.B, "T": shape.T, "C": shape.C, "NH": shape.NH}},
            [part], trimul_flops(shape.B, shape.T, shape.C, shape.NH), [(qkv, qkv_h)], [att])
    if name == "dense_ragged":
        dp, dh, do = dense_part(ds)
        return finish("dense ragged (M=960,I=770,H=768)",
                      {"dense": {"M": ds.M, "I": ds.I, "H": ds.H}},
                      [dp], dense_flops(ds.M, ds.I, ds.H), dh, do)
    if name == "dense_ragged_2304":
        # The ragged layer at the H its page measures (960 x 770 x 2304).
        s2304 = synth.DenseShape(M=ds.M, I=ds.I, H=2304)
        dp, dh, do = dense_part(s2304, traffic=None)
        return finish("dense ragged (M=960,I=770,H=2304)",
                      {"dense": {"M": s2304.M, "I": s2304.I, "H": s2304.H}},
                      [dp], dense_flops(s2304.M, s2304.I, s2304.H), dh, do)
    if name == "dense_sweep":
        gp, gh, go, flops, calls, (I, H, n) = sweep_parts()
        parts = [Part(label, fn, kernel="dense_sm103a_kernel", bound="tensor", per_launch=f)
                 for label, _, f, fn in calls]
        return finish("dense dynamic-shape sweep: 32 calls, M = 16*T, T ~ U{1..128} (seed 0), "
                      "I=768, H=3072", {"dense_sweep": {"calls": n, "I": I, "H": H}},
                      parts, flops, gh, go)
    if name == "dense_sweep_grouped":
        gp, gh, go, flops, calls, (I, H, n) = sweep_parts()
        return finish("dense dynamic-shape sweep, grouped: the same 32 problems (M = 16*T, "
                      "T ~ U{1..128}, seed 0, I=768, H=3072) in one dense_xwt_grouped launch",
                      {"dense_sweep": {"calls": n, "I": I, "H": H, "grouped": True}},
                      [gp], flops, gh, go, calls=calls)
    if name == "bmm_nt":
        bs = synth.BMM_NT_RAGGED
        X_h, W_h = synth.bmm_input(bs, seed=0)
        X, W = X_h.to(dev), W_h.to(dev)
        Y = torch.empty((bs.batch, bs.T1, bs.T2), dtype=torch.float32, device=dev)
        fn = lambda st: csa.batch_matmul_nt(Y, X, W, bs.batch, bs.T1, bs.T2, bs.D, stream=st)
        flops = 2 * bs.batch * bs.T1 * bs.T2 * bs.D
        nbytes = bs.batch * bs.T1 * bs.T2 * 4 + bs.batch * (bs.T1 + bs.T2) * bs.D * 2
        part = Part("bmm_nt", fn, kernel="trimul_sm103a_kernel", bound="hbm", per_launch=nbytes)
        return finish("batched NT product (B*NH=192, T=120, D=64; DietCode BatchMatmulNT)",
                      {"bmm_nt": {"batch": bs.batch, "T1": bs.T1, "T2": bs.T2, "D": bs.D}},
                      [part], flops, [(X, X_h), (W, W_h)], [Y])
    raise ValueError(f"unknown workload {name}")


WORKLOADS = ["step", "step_gpt2", "trimul_gpt2", "trimul_long", "trimul_gpt2_lower",
             "trimul_long_lower", "dense_ragged", "dense_ragged_2304", "dense_sweep",
             "dense_sweep_grouped", "bmm_nt",
             "softmax_gpt2", "softmax_long", "trimul_f32_gpt2", "trimul_f32_long"]


# The pages' own figures for exactly a bench workload (the same useful TFLOP/s on the
# same shape, measured on other GPUs): vs_baseline divides by them, as context.
PAGE_FIGURES = {
    "dense_ragged_2304": (11.6, "DietCode tests/codegen/test_1_local_padding.py, "
                                "test_local_padding: the 960 x 770 x 2304 dense layer with "
                                "local padding, ~11.6 TFLOP/s on an RTX 3090"),
    "bmm_nt": (8.7, "DietCode tests/codegen/test_1_local_padding.py, test_local_padding_ii: "
                    "BatchMatmulNT (B, T, H, NH = 16, 120, 768, 12) padded, ~8.7 TFLOP/s on "
                    "an RTX 3090"),
}


def roofline_entry(part, seconds, hbm_peak, bf16_peak, peak_src, timing):
    """Achieved rate of one kernel launch against its bound's measured peak."""
    if part.bound == "hbm":
        achieved = part.per_launch / seconds / 1e9
        return {"kernel": part.kernel, "part": part.label, "bound": "hbm",
                "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst copy)",
                "algorithmic_bytes_per_launch": part.per_launch,
                "launch_us": round(seconds * 1e6, 2),
                "traffic": recorded_traffic(part.traffic) if part.traffic else None,
                "timing": timing}
    achieved = part.per_launch / seconds / 1e12
    return {"kernel": part.kernel, "part": part.label, "bound": "tensor",
            "achieved": round(achieved, 2), "peak": bf16_peak, "unit": "TFLOP/s",
            "frac": round(achieved / bf16_peak, 4),
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json bf16_tflops, burst cuBLAS)",
            "algorithmic_flops_per_launch": part.per_launch,
            "launch_us": round(seconds * 1e6, 2),
            "traffic": recorded_traffic(part.traffic) if part.traffic else None,
            "timing": timing}


def run_ours(args, rank, world, local):
    import torch

    import causal_attention_score_gb300 as csa
    from causal_attention_score_gb300 import build_lib
    build_lib.build()  # a no-op when the library matches its sources

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = make_workload(args.workload, dev)
    if wl.branches and args.dense_sms is not None:
        # (the first branch holds the dense calls; a limit of 0 lifts theirs)
        wl.branches = [(args.dense_sms if i == 0 else limit, parts)
                       for i, (limit, parts) in enumerate(wl.branches)]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    P = len(wl.parts)

    branch_streams = []
    if wl.branches:
        branch_streams = [torch.cuda.Stream(dev) for _ in wl.branches]
        for (limit, _), bs in zip(wl.branches, branch_streams):
            csa.set_stream_sm_limit(bs, limit)

    def launch(st):
        if wl.branches:
            for bs in branch_streams:
                bs.wait_stream(st)
            for (_, parts), bs in zip(wl.branches, branch_streams):
                for part in parts:
                    part.fn(bs)
            for bs in branch_streams:
                st.wait_stream(bs)
        else:
            for part in wl.parts:
                part.fn(st)

    def step():
        launch(stream)

    graph = None
    graph_error = None
    if args.graph or (wl.branches and not args.direct):
        # The step's launches captured once and replayed as one CUDA graph. A step
        # whose parts run on concurrent streams takes this form by default: the graph
        # holds the fork and the join itself, so the branches overlap however the
        # streams map onto the GPU's hardware queues (direct launches of the default
        # step overlapped only with a short queue and CUDA_DEVICE_MAX_CONNECTIONS=32:
        # 443 us per step; with 200 steps queued they ran one after the other, 635 us;
        # the graph, 439 us).
        step()
        torch.cuda.synchronize(dev)
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(graph, stream=side):
                launch(side)
            torch.cuda.synchronize(dev)
        except Exception as e:  # reported in config.launch; the steps then launch directly
            if args.graph:
                raise
            graph_error = f"{type(e).__name__}: {e}"
            graph = None
            torch.cuda.synchronize(dev)

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        flush.zero_()
        if i == args.warmup - 1:
            w0.record(stream)
        run_step()
    w1.record(stream)
    torch.cuda.synchronize(dev)
    if csa.get_status(stream) != 0:
        raise RuntimeError("device status not ok after warm-up")
    est_ms = max(w0.elapsed_time(w1), 1e-3)

    # Clock soak: the same steps back to back (with their L2 flushes) for about
    # --soak-ms, so that the timed steps run at the clocks a sustained load settles at.
    soak_sampler = ClockSampler(nvml_index(local), period_s=0.0005)
    n_soak = 0
    if args.soak_ms > 0:
        n_soak = max(1, min(20000, int(math.ceil(args.soak_ms / (est_ms + 0.05)))))
        barrier(world)
        torch.cuda.synchronize(dev)
        soak_sampler.start()
        s0 = time.perf_counter()
        for _ in range(n_soak):
            flush.zero_()
            run_step()
        torch.cuda.synchronize(dev)
        soak_wall = time.perf_counter() - s0
        soak_sampler.stop()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    sampler = ClockSampler(nvml_index(local), period_s=0.0005)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    wall0 = time.perf_counter()
    # The timed region: whole steps, one event before and one after each. (An event
    # between two parts would sit between their kernels in the stream and keep the
    # second from starting its launch under the first one's tail.)
    for i in range(K):
        flush.zero_()  # evict L2 between steps; not inside the timed events
        ev[i][0].record(stream)
        run_step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    sampler.stop()
    if csa.get_status(stream) != 0:
        raise RuntimeError("device status not ok after the timed steps")

    # Per-part times (each kernel's launch duration) for a step of several parts: a
    # second pass of K steps, launched directly, with an event after each part.
    part_ms = None
    if P > 1:
        pev = [[torch.cuda.Event(enable_timing=True) for _ in range(P + 1)] for _ in range(K)]
        torch.cuda.synchronize(dev)
        for i in range(K):
            flush.zero_()
            pev[i][0].record(stream)
            for p, part in enumerate(wl.parts):
                part.fn(stream)
                pev[i][p + 1].record(stream)
        torch.cuda.synchronize(dev)
        if csa.get_status(stream) != 0:
            raise RuntimeError("device status not ok after the per-part steps")
        part_ms = [statistics.mean(e[p].elapsed_time(e[p + 1]) for e in pev) for p in range(P)]

    # Separate calls (the sweep's problems one dense_xwt call each): a third pass, L2
    # flushed before each call, an event on either side of it.
    # The event timer advances in steps of about 1 us here, so each call's time is the
    # mean over the repetitions (a median would snap to a step). The same timing around
    # a one-element kernel gives the floor that every call's figure includes.
    call_ms = None
    floor_ms = None
    if wl.calls:
        reps = max(3, min(K, 40))
        one = torch.zeros(1, device=dev)
        fns = [fn for (_, _, _, fn) in wl.calls] + [lambda st: one.add_(1)]
        cev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in fns] for _ in range(reps)]
        for fn in fns:  # (the first launch of a kernel also loads its module)
            fn(stream)
        torch.cuda.synchronize(dev)
        for r in range(reps):
            for c, fn in enumerate(fns):
                flush.zero_()
                cev[r][c][0].record(stream)
                fn(stream)
                cev[r][c][1].record(stream)
        torch.cuda.synchronize(dev)
        if csa.get_status(stream) != 0:
            raise RuntimeError("device status not ok after the separate calls")
        means = [statistics.mean(cev[r][c][0].elapsed_time(cev[r][c][1]) for r in range(reps))
                 for c in range(len(fns))]
        call_ms, floor_ms = means[:-1], means[-1]
    barrier(world)

    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = world * K * wl.flops / (total_ms * 1e-3) / 1e12
    if P == 1:
        part_ms = [statistics.mean(step_ms)]

    # End to end through the public API: host (pinned) inputs in, host results out.
    # Two lanes, each with its own stream and its own device and host buffers,
    # take alternate steps: one lane's results stream back to the host while the
    # other copies its inputs in and computes. Every step still copies all of its
    # inputs in and all of its results out.
    wl2 = make_workload(args.workload, dev)
    lanes = [(wl, torch.cuda.Stream(dev)), (wl2, torch.cuda.Stream(dev))]

    def e2e_step(i):
        lw, ls = lanes[i % 2]
        with torch.cuda.stream(ls):
            for d, h in lw.h2d:
                d.copy_(h, non_blocking=True)
            for part in lw.parts:
                part.fn(ls)
            for h, d in lw.d2h:
                h.copy_(d, non_blocking=True)

    def e2e_run(n, e_start):
        for _, ls in lanes:
            ls.wait_event(e_start)
        for i in range(n):
            e2e_step(i)
        for _, ls in lanes:
            stream.wait_stream(ls)

    e_w = torch.cuda.Event()
    e_w.record(stream)
    e2e_run(max(2, min(args.warmup, 4)), e_w)
    torch.cuda.synchronize(dev)
    ke = max(1, min(K, args.e2e_steps))
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(ke, e0)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    barrier(world)
    if csa.get_status(stream) != 0:
        raise RuntimeError("device status not ok after the end-to-end steps")
    h2d = sum(d.numel() * d.element_size() for d, _ in wl.h2d)
    d2h = sum(d.numel() * d.element_size() for _, d in wl.d2h)
    e2e_value = world * ke * wl.flops / (e2e_ms * 1e-3) / 1e12

    hbm_peak, bf16_peak, peak_src = measured_peaks()
    if P > 1:
        timing = ("CUDA events around its launch, in a second pass of the same K steps "
                  "(direct launches) with an event after each part")
    else:
        timing = "CUDA events around each step of the timed region"
    rooflines = [roofline_entry(part, ms * 1e-3, hbm_peak, bf16_peak, peak_src, timing)
                 for part, ms in zip(wl.parts, part_ms)]
    dominant = max(range(P), key=lambda p: part_ms[p])
    config = {"workload": wl.name, **wl.config,
              "l2": "flushed between timed steps (256 MiB write, outside the timed events)",
              "launch": ("one CUDA graph per step" if graph is not None else
                         "direct launches" + (f" (graph capture failed: {graph_error})"
                                              if graph_error else "")),
              "schedule": ("; ".join(
                  f"stream {i}: {' + '.join(p.label for p in parts)}"
                  + (f" (at most {limit} SMs)" if limit else " (no SM limit)")
                  for i, (limit, parts) in enumerate(wl.branches))
                  + "; launched in this order, forked from and joined into the step's stream"
                  if wl.branches else "the parts one after another on one stream"),
              "parallelism": f"replicas x{world}"}
    clocks = sampler.summary()
    if n_soak:
        soak = soak_sampler.summary()
        soak.update({"steps": n_soak, "wall_s": round(soak_wall, 4)})
        clocks["soak"] = soak
    result = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (round(value / PAGE_FIGURES[args.workload][0], 3)
                        if args.workload in PAGE_FIGURES else None),
        "dtype": wl.dtype,
        "data": wl.data,
        "config": config,
        "pct_of_bf16_peak": round(100 * value / world / bf16_peak, 3),
        "roofline": rooflines[dominant],
        "rooflines": rooflines,
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": ke,
                "ms_per_step": round(e2e_ms / ke, 4),
                "pipeline": "two lanes (stream + buffers each) take alternate steps; each step "
                            "copies its inputs in and its results out"},
        "gpu_launches": wl.kernels_per_step * K,
        "flops_per_step": wl.flops,
        "ms_step_percentiles": {f"p{q}": round(_percentile(step_ms, q), 5) for q in (10, 50, 90)},
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
    }
    if args.workload in PAGE_FIGURES:
        result["vs_baseline_source"] = PAGE_FIGURES[args.workload][1]
    if wl.parts and all(p.hbm_bytes for p in wl.parts):
        # The whole step against HBM: every part's algorithmic bytes over the step time.
        step_bytes = sum(p.hbm_bytes for p in wl.parts)
        achieved = step_bytes / (total_ms / K * 1e-3) / 1e9
        result["step_roofline"] = {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "algorithmic_bytes_per_step": step_bytes,
            "note": "all parts' algorithmic bytes (inputs read once, outputs written once) "
                    "over the step time"}
    if P <= 40:
        result["parts"] = {f"{part.label}_us": round(ms * 1e3, 2)
                           for part, ms in zip(wl.parts, part_ms)}
        if P > 1:
            result["parts_timing"] = ("a second pass of the K steps, direct launches, with an "
                                      "event after each part")
    if call_ms is not None:
        result["sweep_calls"] = {
            "timing": "each problem as its own dense_xwt call, L2 flushed before each, mean "
                      "over the repetitions of CUDA events around the call",
            "reps": max(3, min(K, 40)),
            "timing_floor_us": round(floor_ms * 1e3, 2),
            "timing_floor": "the same timing around a one-element torch kernel",
            "total_us": round(sum(call_ms) * 1e3, 2),
            "calls": [{"M": M, "us": round(ms * 1e3, 2),
                       "frac_bf16": round(f / (ms * 1e-3) / 1e12 / bf16_peak, 4)}
                      for (_, M, f, _), ms in zip(wl.calls, call_ms)]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload in ORACLE_SAMPLES:
        result["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    return result


# --------------------------------------------------------- oracle timing --

class OracleSample:
    """Bounded samples of a step on the oracle. Sample i covers one (b, h) head of the
    score product (all its rows) and the rows r = i (mod 32) of each dense problem, so
    that 32 consecutive samples of the default step cover about one whole step."""

    def __init__(self, workload):
        import numpy as np

        from causal_attention_score_gb300 import synth
        self.np = np
        ts = synth.TRIMUL_LONG if workload == "step" else synth.TRIMUL_GPT2
        self.ts = ts
        self.qkv = synth.bf16_bits(synth.trimul_input(ts, seed=0, dist="normal")).reshape(-1)
        X, W = synth.dense_input(synth.DENSE_RAGGED, seed=0)
        self.dense = [(synth.bf16_bits(X).reshape(-1), synth.bf16_bits(W).reshape(-1),
                       synth.DENSE_RAGGED.M, synth.DENSE_RAGGED.I, synth.DENSE_RAGGED.H)]
        self.sweep = workload == "step"
        if self.sweep:
            xs, Ws = synth.dense_sweep_inputs(seed=0)
            wb = synth.bf16_bits(Ws).reshape(-1)
            H, I = Ws.shape
            self.dense += [(synth.bf16_bits(Xi).reshape(-1), wb, Xi.shape[0], I, H) for Xi in xs]
        self.stride = 32

    def describe(self):
        if self.sweep:
            return ("one (b,h) head of trimul long context (4096 rows) + rows r = i mod 32 of "
                    "each of the 33 dense problems (the sweep's 32 and the ragged one): 1/32 of "
                    "a step")
        return "one (b,h) head of trimul GPT-2 (1024 rows) + 64 rows of dense ragged"

    def parts(self, i):
        """What sample i computes: the (b, h, t) rows of the score product and, per dense
        problem, its rows; with the useful flops of each."""
        np = self.np
        ts = self.ts
        bh = i % (ts.B * ts.NH)
        b, h = divmod(bh, ts.NH)
        bht = np.array([(b, h, t) for t in range(ts.T)], dtype=np.int64)
        dense = []
        for xb, wb, M, I, H in self.dense:
            if self.sweep:
                rows = np.arange(i % self.stride, M, self.stride, dtype=np.int64)
            else:
                rows = (np.arange(64, dtype=np.int64) + 64 * i) % M
            dense.append((xb, wb, M, I, H, rows))
        return bht, 2 * ts.HS * ts.T * (ts.T + 1) // 2, dense

    def flops(self, i):
        _, f, dense = self.parts(i)
        return f + sum(2 * int(rows.size) * I * H for _, _, _, I, H, rows in dense)

    def __call__(self, o, i):
        """Runs sample i on oracle `o`; returns its useful flops."""
        ts = self.ts
        bht, _, dense = self.parts(i)
        o.trimul_rows(self.qkv, ts.B, ts.T, ts.C, ts.NH, bht)
        for xb, wb, M, I, H, rows in dense:
            if rows.size:
                o.dense_rows(xb, wb, M, I, H, rows)
        return self.flops(i)


ORACLE_SAMPLES = ("step", "step_gpt2")


def cpu_baseline(workload: str, seconds: float):
    """The oracle as it stands on the host cores: repeated bounded samples of the step for
    about `seconds` of CPU time; throughput in the metric's unit."""
    import oracle
    o = oracle.get()
    sample = OracleSample(workload)
    flops, i = 0, 0
    t0 = time.perf_counter()
    while True:
        flops += sample(o, i)
        i += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    cores = o.num_threads()
    # The same samples on one thread, for about a quarter of the time (at least one).
    o.set_num_threads(1)
    try:
        flops1, j = 0, 0
        t1 = time.perf_counter()
        while True:
            flops1 += sample(o, j)
            j += 1
            if time.perf_counter() - t1 >= seconds / 4:
                break
        dt1 = time.perf_counter() - t1
    finally:
        o.set_num_threads(cores)
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{i} samples, each {sample.describe()}; fp64, {dt:.1f} s",
            "value_1thread": round(flops1 / dt1 / 1e12, 6),
            "sample_1thread": f"{j} of the same samples on 1 thread, {dt1:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    o = oracle.get()
    workload = args.workload if args.workload in ORACLE_SAMPLES else "step"
    sample = OracleSample(workload)
    for i in range(args.warmup):
        sample(o, i)
    flops = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops += sample(o, i)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    names = {"step": "trimul long context (B=2,T=4096,C=2048,NH=16,HS=128) + dense dynamic-shape "
                     "sweep (32 problems M=16*T, T~U{1..128} seed 0, I=768, H=3072) + dense "
                     "ragged (M=960,I=770,H=768)",
             "step_gpt2": "trimul GPT-2-small (B=8,T=1024,C=768,NH=12,HS=64) + dense ragged "
                          "(M=960,I=770,H=768)"}
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded, rounded to bf16)",
        "config": {"workload": names[workload] + "; each step a bounded sample: "
                   + sample.describe()},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": o.num_threads(),
                         "kind": "oracle", "sample": "per step: " + sample.describe()},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--soak-ms", type=float, default=150.0,
                   help="run the step back to back this long before the timed region")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--workload", choices=WORKLOADS, default="step",
                   help="what a step runs (default: the headline step)")
    p.add_argument("--graph", action="store_true",
                   help="capture each step's launches as one CUDA graph and replay it (the "
                        "default for a step whose parts run on concurrent streams)")
    p.add_argument("--dense-sms", type=int, default=None,
                   help=f"SM limit of the dense calls' stream in a step with concurrent "
                        f"streams (default: {STEP_DENSE_SMS} in the default step; 0: none)")
    p.add_argument("--direct", action="store_true",
                   help="launch every step's kernels directly, even on concurrent streams")
    args = p.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        p.error("--warmup must be >= 3")
    if args.graph and args.direct:
        p.error("--graph and --direct exclude each other")

    if args.impl == "reference":
        # The oracle runs on the host of rank 0 only; other ranks have no work.
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        res = run_reference(args, rank, world)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
        return
    rank, world, local = dist_setup(args.gpus)
    res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
