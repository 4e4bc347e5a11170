"""The bench's multi-rank host logic on CPU, two gloo ranks: each rank runs its own
replica of the decode workload (its own requests), and the whole-job number is the
units of all ranks over the slowest rank's time. No GPU and no collective on the data
path; the only collectives are the timing reductions tested here."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from dsa_sparse_attention_02_gb300 import inputs

# per-rank (units, ms): unequal on purpose, so a sum taken where a max belongs (or the
# other way round) changes the result
RANK_WORK = [(64 * 20, 12.5), (96 * 20, 17.0)]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        units, ms = RANK_WORK[rank]
        value, ms_max = bench.aggregate_over_ranks(units, ms, dist, "cpu")
        out[rank] = (value, ms_max)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    units = sum(u for u, _ in RANK_WORK)
    slowest = max(ms for _, ms in RANK_WORK)
    for r in range(world):
        value, ms_max = out[r]
        assert ms_max == slowest
        assert value == pytest.approx(units / (slowest / 1000.0), rel=1e-12)


def test_aggregate_single_rank_is_plain_rate():
    value, ms = bench.aggregate_over_ranks(640, 8.0)
    assert ms == 8.0 and value == pytest.approx(80000.0)


def test_replicas_draw_their_own_requests():
    seeds = [bench.replica_seed(r) for r in range(8)]
    assert len(set(seeds)) == 8
    assert seeds[0] == inputs.CONFIG_SEEDS["decode"]     # rank 0 is the single-GPU workload
    a, b = (inputs.make_config("decode", batch=4, ctx_scale=1 / 16, seed=s) for s in seeds[:2])
    assert not np.array_equal(a.seq_lens, b.seq_lens)
