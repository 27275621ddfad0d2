"""The N > 1 host logic of bench.py on CPU: two gloo ranks (world size 2) as child
processes. Each rank reports a different elapsed time; both must agree on the slowest
rank's, the whole-job rate must count both replicas' work over that time, and only
rank 0 may print. The reference arm must do nothing on ranks other than 0."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["ROOT"])
import torch, torch.distributed as dist
import bench
rank, world, local = bench._rank()
dist.init_process_group("gloo", init_method="env://")
elapsed = 10.0 + 5.0 * rank            # rank 1 is the slower one
got = bench.max_over_ranks(elapsed, world)
rate = bench.job_rate(1000, 20, world, got)
if rank == 0:
    print(json.dumps({"elapsed": got, "rate": rate}))
dist.barrier()
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(code, world=2):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, ROOT=ROOT, RANK=str(r), WORLD_SIZE=str(world), LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e[-2000:]
    return [o for o, _ in outs]


def test_max_over_ranks_and_job_rate_world2():
    out0, out1 = _run_ranks(CHILD)
    assert out1.strip() == ""  # only rank 0 prints
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["elapsed"] == 15.0  # the slowest rank's time, on every rank
    assert abs(line["rate"] - 1000 * 20 * 2 / 0.015) < 1e-6  # both replicas' work


def test_reference_arm_idle_on_other_ranks():
    code = r"""
import os, sys
sys.path.insert(0, os.environ["ROOT"])
import bench, argparse
bench.run_reference(argparse.Namespace(steps=1, warmup=0, K=8, V=151936, T=1.0, B=64))
print("done")
"""
    env = dict(os.environ, ROOT=ROOT, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == "done"  # returned at once: no JSON line, no work
