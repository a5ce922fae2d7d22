"""bench.py's multi-process handling on the CPU: two ranks over gloo on
127.0.0.1 (the launch torchrun performs), checking the barrier, the
max-over-ranks reduction the step time goes through, and that only rank 0
runs and prints the reference arm."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import bench
world, rank, local = bench.dist_setup(2)
bench.barrier(world)
m = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
bench.barrier(world)
print(json.dumps({"rank": rank, "world": world, "max": m}))
import torch.distributed as dist
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, port):
    env = dict(os.environ)
    env.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    return env


def test_two_gloo_ranks_reduce_the_step_time_to_its_maximum():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", RANK_SCRIPT, ROOT], env=_env(r, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=180)
            assert p.returncode == 0, err[-2000:]
            outs.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["world"] == 2 and o["max"] == 15.0 for o in outs)


def test_reference_arm_runs_on_rank_zero_only():
    env = _env(1, _free_port())
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
