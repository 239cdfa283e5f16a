"""Host logic of the multi-GPU bench run, on CPU ranks with the gloo backend.

Each rank of `bench.py --gpus N` runs an independent replica (its own batch, no
collective on the data path); the only exchange is the max over ranks of the timed
durations, and the whole-job throughput counts every rank's work.  These tests run
that exchange on two gloo ranks and check the reference arm's rank gating.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r was slow in a different stage: the reported times are the per-stage maxima
        local = [10.0 + rank, 5.0 - rank, 1.5 * (rank + 1)]
        reduced = bench.max_over_ranks(local, "cpu")
        seed = bench.rank_seed("bf16_train", rank)
        # the reference arm: only rank 0 runs the oracle and prints; the others return at once
        out = io.StringIO()
        if rank != 0:
            from joint_sequence_depth_gb300.inputs import WORKLOADS

            args = type("A", (), {"steps": 1, "warmup": 0, "gpus": world})()
            with redirect_stdout(out):
                rc = bench.run_reference(args, WORKLOADS["bf16_train"])
        else:
            rc = 0
        results[rank] = (reduced, seed, rc, out.getvalue())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_gate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, results), nprocs=world, join=True, start_method="spawn")
        res = dict(results)
    assert sorted(res) == [0, 1]
    for rank in range(world):
        reduced, _, rc, out = res[rank]
        assert reduced == [11.0, 5.0, 3.0]  # element-wise max over the two ranks
        assert rc == 0
    assert res[0][1] != res[1][1]  # independent batches per rank
    assert res[1][3] == ""  # rank 1 of the reference arm printed nothing


def test_aggregate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    one = bench.aggregate_tflops(2.0e12, 1000.0, 1)
    assert one == pytest.approx(2.0)
    assert bench.aggregate_tflops(2.0e12, 1000.0, 4) == pytest.approx(4 * one)
    # without an initialised process group the reduction is the identity
    assert bench.max_over_ranks([3, 1.5], "cpu") == [3.0, 1.5]
