"""The multi-process side of bench.py, on CPU with the gloo backend (world size 2).

The layer shards by tokens with no exchange, so N GPUs run N independent replicas: each rank
times its own steps, the ranks meet at a barrier on both sides of the timed region, and the
reported time is the maximum over ranks. These tests check that host logic without a GPU:
the barrier and the max-over-ranks reduction of bench.py in two gloo processes, and the
reference arm launched the way the multi-GPU run launches it (torch.distributed.run, two
ranks), where rank 0 alone prints one JSON line and both ranks exit 0."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    r, w, _ = bench.dist_setup()
    assert (r, w) == (rank, world)
    bench.barrier()
    # rank r "measured" 1 + r ms: every rank must report the slowest
    got = bench.max_over_ranks(1.0 + rank)
    bench.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got}, f)
    torch.distributed.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    vals = [json.load(open(tmp_path / f"rank{r}.json"))["max"] for r in range(2)]
    assert vals == [2.0, 2.0]


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "3", "--warmup", "1", "--workload", "tiny_T8"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
