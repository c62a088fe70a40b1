"""The bench's multi-GPU host logic on CPU: world size 2 over gloo.

Replicas only (no data-path collective): each rank runs the same per-GPU
workload, the job's time is the slowest rank's (an all-reduce MAX), the
value is the whole job's throughput, and only rank 0 prints.  These run
without a GPU: the gloo backend and CPU tensors stand in for NCCL and
device tensors."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    import torch
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(values[rank], dist, torch.device("cpu"))
        out[rank] = got
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    values = [3.25, 7.5]
    mp.start_processes(_rank_main, args=(2, _free_port(), values, out), nprocs=2,
                       start_method="spawn", join=True)
    assert out[0] == 7.5 and out[1] == 7.5


def test_whole_job_value_is_weak_scaling():
    import bench
    # every rank processes 1e9 bytes in 0.5 s: the job moves 2e9 bytes in 0.5 s
    assert bench.whole_job_value(1e9, 2, 0.5, 1e-9) == pytest.approx(4.0)
    assert bench.max_over_ranks(1.5, None, None) == 1.5


def test_reference_arm_prints_on_rank_zero_only():
    outs = []
    procs = []
    for rank in (0, 1):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1")
        procs.append(subprocess.Popen(
            [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
             "--steps", "1", "--warmup", "3", "--ref-step-seconds", "0.02"],
            cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    for p in procs:
        o, e = p.communicate(timeout=300)
        assert p.returncode == 0, e
        outs.append(o.strip())
    line = json.loads(outs[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert outs[1] == ""
