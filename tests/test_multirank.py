"""The benchmark's multi-rank path on CPU: two gloo ranks agree on the job time
(max over ranks) and the reference arm runs on rank 0 only."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import bench, torch.distributed as dist
rank, world, local = bench.dist_setup(2)
t = 1.0 + rank  # rank 1 is slower
m = bench.max_over_ranks(t, world)
bench.barrier(world)
with open(os.path.join({out!r}, f"rank{{rank}}.txt"), "w") as f:
    f.write(f"{{rank}} {{world}} {{m}}")
dist.destroy_process_group()
"""


def _run_two(code, extra_env=None):
    env = dict(os.environ, CSA_BENCH_BACKEND="gloo")
    env.update(extra_env or {})
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29517", "-c", code]
    return subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=240, cwd=ROOT)


def test_two_gloo_ranks_take_max_time(tmp_path):
    script = tmp_path / "w.py"
    script.write_text(WORKER.format(root=ROOT, out=str(tmp_path)))
    env = dict(os.environ, CSA_BENCH_BACKEND="gloo")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29517", str(script)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=240, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    for rank in (0, 1):
        got_rank, world, m = (tmp_path / f"rank{rank}.txt").read_text().split()
        assert int(got_rank) == rank and int(world) == 2 and float(m) == 2.0


def test_reference_arm_runs_on_rank0_only(tmp_path):
    env = dict(os.environ)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29518",
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "2",
           "--warmup", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = lines[0]
    assert res["impl"] == "reference" and res["value"] > 0 and res["unit"] == "TFLOP/s"
    assert res["cpu_baseline"]["kind"] == "oracle"
    assert res["e2e"]["h2d_bytes_per_step"] == 0
