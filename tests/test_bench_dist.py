"""bench.py's multi-rank host logic, on CPU with two gloo ranks.

Under torchrun every rank verifies its own batch (weak scaling), the timed
region of a step is the slowest rank's, the whole-job value counts every
rank's positions, and the reference arm prints one line from rank 0 only.
No GPU is involved: the collectives run on the gloo backend.
"""
import contextlib
import io
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        cpu = torch.device("cpu")
        local_ms = [1.5, 2.5][rank]                     # rank 1 is the slow one
        ms = bench.reduce_max(local_ms, dist, cpu)
        te = bench.reduce_max([0.25, 0.125][rank], dist, cpu)
        out = io.StringIO()
        args = bench.parse(["--impl", "reference", "--config", "chain_b1_k4_v1024_f32",
                            "--steps", "2", "--warmup", "1"])
        with contextlib.redirect_stdout(out):
            bench.run_reference(args, rank, WORLD)
        dist.barrier()
        q.put((rank, ms, te, out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_report():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    mp.start_processes(_rank, args=(_free_port(), q), nprocs=WORLD, start_method="spawn")
    got = sorted(q.get() for _ in range(WORLD))
    for rank, ms, te, text in got:
        assert ms == 2.5, "the step time is the slowest rank's"
        assert te == 0.25
        lines = [ln for ln in text.splitlines() if ln.strip()]
        if rank == 0:
            assert len(lines) == 1 and '"impl": "reference"' in lines[0] and '"n_gpus": 2' in lines[0]
        else:
            assert lines == [], "only rank 0 prints"


def test_job_throughput_counts_every_rank():
    # 448 positions per rank per step, 2 ranks, the slowest step 0.05 ms
    assert bench.job_throughput(2, 448, 0.05) == pytest.approx(2 * 448 / 0.05e-3)
    assert bench.job_throughput(1, 448, 0.05) * 2 == pytest.approx(bench.job_throughput(2, 448, 0.05))
    assert bench.reduce_max(3.0, None, None) == 3.0


def test_each_rank_draws_its_own_batch():
    seeds = [bench.rank_seed(0, r) for r in range(4)]
    assert len(set(seeds)) == 4
    a = workloads.make("chain_b1_k4_v1024_f32", seed=seeds[0])
    b = workloads.make("chain_b1_k4_v1024_f32", seed=seeds[1])
    assert not np.array_equal(a["target"], b["target"])
    assert a["target"].shape == b["target"].shape  # same shape: weak scaling
