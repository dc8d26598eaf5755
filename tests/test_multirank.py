"""Multi-rank host logic of bench.py, run as two gloo ranks on the CPU.

The path shards over independent (batch, head) replicas, one process per GPU, with
no collective on the data path: what runs across ranks is the rendezvous, the
barriers around the timed region, the maximum over ranks of the step time and the
whole-job throughput that rank 0 prints.  The reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_CODE = r"""
import json, os, sys
sys.path.insert(0, os.environ["FBD_ROOT"])
import bench
world = int(os.environ["WORLD_SIZE"]); rank = int(os.environ["RANK"])
bench.dist_init(world, backend="gloo")
bench.barrier(world)
ms = [4.0, 5.5][rank]
slowest = bench.max_over_ranks(ms, world)
value = bench.job_tflops(2.0e12, world, slowest)
bench.barrier(world)
import torch.distributed as dist
dist.destroy_process_group()
print(json.dumps({"rank": rank, "slowest": slowest, "value": value}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), FBD_ROOT=ROOT)
    return env


def test_two_gloo_ranks_agree_on_the_slowest_step_and_the_job_throughput():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", RANK_CODE], env=_env(r, 2, port), cwd=ROOT,
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE) for r in range(2)]
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=180)
            assert p.returncode == 0, err.decode()[-2000:]
            outs.append(json.loads(out.decode().strip().splitlines()[-1]))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["slowest"] == 5.5
        # 2 ranks x 2 TFLOP each, in the slowest rank's 5.5 ms
        assert abs(o["value"] - 2 * 2.0 / 5.5e-3) < 1e-9


def test_job_throughput_single_rank_is_the_plain_rate():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert abs(bench.job_tflops(1.0e12, 1, 2.0) - 500.0) < 1e-9


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the other ranks of the reference arm exit 0 at once, printing nothing."""
    env = _env(1, 2, _free_port())
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1"],
                       env=env, cwd=ROOT, capture_output=True, timeout=180)
    assert r.returncode == 0, r.stderr.decode()[-2000:]
    assert r.stdout.decode().strip() == ""
