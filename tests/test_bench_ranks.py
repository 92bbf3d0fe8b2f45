"""The benchmark's multi-rank logic on CPU (gloo, world size 2): the maximum
over ranks, and the reference arm that runs on rank 0 only and prints one
JSON line.  Each rank is a separate process launched by torch's launcher on
127.0.0.1."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _torchrun(args, timeout=240):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(29500 + os.getpid() % 1000)] + args
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_max_over_ranks_with_gloo(tmp_path):
    # each rank writes its result to its own file: the ranks' stdout streams
    # interleave
    script = tmp_path / "ranks.py"
    script.write_text(
        "import os, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import bench\n"
        "world, rank, local = bench.dist_setup(2)\n"
        "m = bench.max_over_ranks(float(rank + 1) * 10.0, world)\n"
        "bench.barrier(world)\n"
        f"open(os.path.join({str(tmp_path)!r}, 'rank%d.txt' % rank), 'w').write(repr(m))\n"
        "import torch.distributed as dist; dist.destroy_process_group()\n")
    r = _torchrun([str(script)])
    assert r.returncode == 0, r.stderr[-2000:]
    got = [float((tmp_path / f"rank{i}.txt").read_text()) for i in range(2)]
    assert got == [20.0, 20.0]


def test_reference_arm_prints_once_from_rank_zero():
    r = _torchrun(["bench.py", "--impl", "reference", "--workload", "tiny", "--gpus", "2",
                   "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
