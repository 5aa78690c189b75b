"""The benchmark's multi-rank plumbing on CPU: world size 2 over gloo
(127.0.0.1).  Each rank is an independent replica; the slowest rank's time
sets the whole job's rate, and only rank 0 runs the reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    assert torch.distributed.get_backend() == "gloo"
    bench.barrier(w)
    # each rank's own elapsed time; the job's time is the slowest rank's
    slowest = bench.max_over_ranks(100.0 + 7.0 * rank, w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"slowest": slowest}, f)
    bench.barrier(w)
    torch.distributed.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time(tmp_path):
    mp.spawn(_rank, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert json.load(open(tmp_path / f"rank{r}.json"))["slowest"] == 107.0


@pytest.mark.parametrize("workload", ["bf16_8192", "transpose_f32_16384", "conv3x3_bf16_32x56x56x256"])
def test_reference_arm_runs_on_rank_zero_only(workload):
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                          "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""
