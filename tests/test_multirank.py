"""The multi-rank harness of bench.py on CPU, world size 2 over gloo.

The path shards by (sequence, kv head) with no collective, so N GPUs run N
independent replicas; the only cross-rank steps are the harness's barrier,
the max of the timed intervals and the sum of the tokens. These run here on
CPU ranks, and the reference arm is checked to print one line from rank 0
only.
"""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist = bench.init_dist(w)
    try:
        bench.barrier(dist)
        mx = bench.max_over_ranks(dist, 10.0 + rank)      # per-rank timed interval
        tot = bench.sum_over_ranks(dist, 100.0 * (rank + 1))  # per-rank tokens
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"max": mx, "sum": tot}, f)
    finally:
        dist.destroy_process_group()


def test_harness_reductions_two_gloo_ranks(tmp_path):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        with open(tmp_path / f"r{rank}.json") as f:
            got = json.load(f)
        assert got == {"max": 11.0, "sum": 300.0}  # every rank sees the job-wide values


def test_reference_arm_rank0_only():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--workload", "tiny_f32", "--steps", "2", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "draft tokens/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
