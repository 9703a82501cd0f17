"""The multi-rank host logic of bench.py on CPU: two gloo ranks (replicas, no data-path collective).

bench.py under torchrun gives every rank its own batch (weak scaling); the ranks meet only to
combine the timings.  The whole-job time is the slowest rank's and the processed units are the sum
over ranks.  This runs that very function over a world of 2 on the gloo backend.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    w, r, lr = bench.dist_setup()
    assert (w, r, lr) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: 10 + r ms for K steps, e2e 3 + 2r ms, units 1000 * (r + 1)
        res = bench.aggregate_over_ranks(torch, 10.0 + rank, 3.0 + 2 * rank, 1000.0 * (rank + 1), 7.0 * (rank + 1),
                                         torch.device("cpu"))
        out[rank] = res
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this multi-threaded process
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        total_ms, e2e_ms, units, e2e_units = res[r]
        assert total_ms == 11.0 and e2e_ms == 5.0        # the slowest rank's times
        assert units == 3000.0 and e2e_units == 21.0     # summed over the replicas


def test_dist_setup_defaults_to_one_rank(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup() == (1, 0, 0)
