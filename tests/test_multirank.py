"""The N > 1 launch path on the CPU (no GPU): two ranks over gloo.

The attention path shards by (batch row, kv head) with no exchange step, so
several GPUs run replicas: each rank times its own steps, the job's time is
the largest over the ranks, and rank 0 alone prints the result line. These
tests run that logic as two host processes: the max-over-ranks reduction the
bench uses, and the bench's reference arm under torchrun (rank 0 prints one
line, the other rank exits 0 without work).
"""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, timings):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max(timings[rank], dist)
        assert got == max(timings), (rank, got)
        assert bench.reduce_max(timings[rank], None) == timings[rank]
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    mp.start_processes(_rank_main, args=(2, _free_port(), [1.25, 3.5]), nprocs=2,
                       start_method="spawn", join=True)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    # one timed step of the default workload's bounded oracle sample (a few seconds of CPU)
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    proc = subprocess.run(
        [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
         "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
         os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
         "--warmup", "0"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert proc.returncode == 0, proc.stderr[-3000:]
    lines = [ln for ln in proc.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, proc.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["steps"] == 1
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0

