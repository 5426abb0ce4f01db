"""The N > 1 bench path on CPU: two gloo ranks exchange timings the way bench.py
does under torchrun (barrier, max over ranks for time, sum over ranks for work)
and the reference arm prints from rank 0 only."""

import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, os.environ["ROOT"])
import bench
world, rank, local = bench.dist_setup()
bench.barrier(world)
t = bench.max_over_ranks(10.0 + rank, world)
w = bench.sum_over_ranks(100.0 * (rank + 1), world)
# one file per rank: two processes printing to one pipe at once can interleave lines
with open(os.path.join(os.environ["OUT_DIR"], f"rank{rank}.json"), "w") as f:
    json.dump({"rank": rank, "world": world, "max": t, "sum": w}, f)
import torch.distributed as dist
dist.destroy_process_group()
"""


def _free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _torchrun(script_args, port, env_extra=None, timeout=240):
    port = _free_port()
    env = dict(os.environ, ROOT=ROOT, CUDA_VISIBLE_DEVICES="")
    if env_extra:
        env.update(env_extra)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}"] + script_args
    return subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=timeout, cwd=ROOT)


def test_two_gloo_ranks_reduce_timings(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER)
    res = _torchrun([str(script)], 29611, env_extra={"OUT_DIR": str(tmp_path)})
    assert res.returncode == 0, res.stderr[-2000:]
    import json
    lines = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(2)]
    assert sorted(l["rank"] for l in lines) == [0, 1]
    for l in lines:
        assert l["world"] == 2 and l["max"] == 11.0 and l["sum"] == 300.0


def test_reference_arm_prints_from_rank_zero_only():
    res = _torchrun([os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
                     "--warmup", "3"], 29612, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1 and '"impl": "reference"' in lines[0]
