"""The multi-GPU path of bench.py is replicas only: every rank runs its own
round on its own seeded inputs, and the job's throughput is all ranks' units
over the slowest rank's time. These tests run that host logic with two gloo
ranks on the CPU (no GPU, no NCCL)."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from speculative_decoding_draft_depth_gb300 import synth
    try:
        # a slower rank 1: every rank must see its time
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        seed = bench.rank_seed(synth.config("batch64").seed, rank)
        cfg = synth.config("tiny", seed=seed)
        z = synth.draw_round_inputs(cfg)["draft_logits"]
        out[rank] = (ms, seed, float(z.ravel()[:64].sum()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_and_draw_their_own_inputs():
    world = 2
    with mp.get_context("spawn").Manager() as m:  # no fork of this (threaded) process
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0       # max over ranks, on every rank
    assert res[0][1] != res[1][1]               # each replica has its own seed
    assert res[0][2] != res[1][2]               # ... and so its own inputs


def test_job_throughput_and_single_process():
    import bench
    # two ranks, 100 rounds each, the slowest took 50 ms: 4000 rounds/s
    assert bench.job_throughput(2, 100, 50.0) == pytest.approx(4000.0)
    assert bench.job_throughput(1, 100, 50.0) == pytest.approx(2000.0)
    # one process: its own time
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
