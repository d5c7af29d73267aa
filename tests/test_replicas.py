"""Replica logic of the benchmark on CPU processes (gloo, world size 2).

The verification path shards over the batch with no exchange, so several GPUs
run independent replicas: each rank verifies its own seeded batch, the
reported time is the slowest rank's, and the rate counts every rank's work.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from workloads import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        spec = synth.with_sizes(synth.SPECS["sampling_chain_b32_g8_v32000_bf16"], B=2, V=257)
        w = synth.make(spec, seed=bench.replica_seed(7, rank))
        ms = [3.0, 5.0][rank]
        slowest = bench.max_over_ranks(ms, dist, torch.device("cpu"))
        rate = bench.whole_job_rate(bench.draft_tokens_per_call(w), world, slowest)
        out[rank] = (slowest, rate, int(w["tokens"].sum()))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_all_work():
    world = 2
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    (ms0, rate0, tok0), (ms1, rate1, tok1) = out[0], out[1]
    assert ms0 == ms1 == 5.0
    assert rate0 == rate1 == pytest.approx(2 * 16 / 5e-3)  # B=2, gamma=8 drafts per replica
    assert tok0 != tok1  # every replica verifies its own batch


def test_single_process_needs_no_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.0, None, "cpu") == 4.0
    assert bench.replica_seed(3, 0) == 3
