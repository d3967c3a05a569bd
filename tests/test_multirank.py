"""The N > 1 host logic of bench.py on CPU ranks (gloo, world size 2).

Every matrix's Muon step is independent, so N GPUs run N replicas with no
collective on the data path; the only cross-rank steps are the barrier around
the timed region and the max over ranks of its duration.  These tests run that
reduction and the whole-job aggregation across two gloo processes.
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = [12.5, 30.25][rank]
        dist.barrier()
        ms = bench.max_over_ranks(ms_local, dist, "cpu")
        out[rank] = (ms, bench.job_tflops(world, 2.5e13, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_on_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, value = res[rank]
        assert ms == 30.25                       # every rank sees the slowest rank's time
        assert value == pytest.approx(2 * 2.5e13 / 30.25e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(7.0) == 7.0
    assert bench.job_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)
