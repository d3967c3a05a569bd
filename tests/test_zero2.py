"""The ZeRO-2-style sharded step: ownership (muon_partition, C, host only) and
the three-phase driver (pretraining_optimizer_step_b300.zero2) on two gloo
ranks on the CPU, with the fp64 oracle as the per-matrix update."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import pretraining_optimizer_step_b300 as mu
import workloads


def work(shape):
    m, n = min(shape), max(shape)
    return 3 * m * m * n + m ** 3


@pytest.mark.parametrize("name,world", [("d2", 2), ("d12", 3), ("d26", 8), ("sweep_512_tall", 5)])
def test_partition_balances_work(name, world):
    shapes = workloads.config_shapes(name)
    owner = mu.muon_partition(shapes, world)
    assert owner == mu.muon_partition(shapes, world)  # deterministic
    assert set(owner) <= set(range(world))
    load = [0] * world
    for s, r in zip(shapes, owner):
        load[r] += work(s)
    # greedy largest-first: the spread is at most one matrix's work
    assert max(load) - min(load) <= max(work(s) for s in shapes)


def test_partition_edge_cases():
    assert mu.muon_partition([(64, 64)] * 3, 1) == [0, 0, 0]
    assert mu.muon_partition([(64, 64), (128, 128)], 4)[1] == 0  # the largest goes first, to rank 0
    assert mu.muon_partition([], 2) == []
    with pytest.raises(mu.MuonError):
        mu.muon_partition([(64, 64)], 0)
    with pytest.raises(mu.MuonError):
        mu.muon_partition([(60, 64)], 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


HYPER = dict(lr=0.02, beta=0.95, nesterov=True, ns_steps=3)


def oracle_compute(params, grads, moms, lr, beta, nesterov, ns_steps):
    for p, g, m in zip(params, grads, moms):
        p1, m1, _ = oracle.muon_matrix(p.numpy(), g.numpy(), m.numpy(), lr=np.float32(lr), beta=np.float32(beta),
                                       nesterov=nesterov, ns_steps=ns_steps)
        p.copy_(torch.from_numpy(p1))
        m.copy_(torch.from_numpy(m1))


SHAPES = [(64, 64), (128, 64), (64, 128), (96, 96), (64, 64), (32, 160)]


def _rank_grads(rank, step):
    return [workloads.make_grad("zero2", 100 * rank + i, s, "cpu", 0, step) for i, s in enumerate(SHAPES)]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        params = [workloads.make_param("zero2", i, s, "cpu", 0) for i, s in enumerate(SHAPES)]
        sharded = mu.zero2.ShardedMuon(params, compute=oracle_compute)
        for step in range(2):
            sharded.step(_rank_grads(rank, step), **HYPER)
        out[rank] = ([p.numpy().copy() for p in params], sharded.owner,
                     {i: m.numpy().copy() for i, m in sharded.momentum.items()})
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_match_one_process_on_the_mean_gradient():
    world = 2
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    # every rank ends with the same weights
    for a, b in zip(res[0][0], res[1][0]):
        assert np.array_equal(a, b)
    owner = res[0][1]
    assert sorted(set(owner)) == [0, 1]
    # reference: one process, the mean of the ranks' gradients, full momentum
    params = [workloads.make_param("zero2", i, s, "cpu", 0).numpy() for i, s in enumerate(SHAPES)]
    moms = [np.zeros(s, np.float32) for s in SHAPES]
    for step in range(2):
        g = [(a + b) * np.float32(0.5) for a, b in zip((t.numpy() for t in _rank_grads(0, step)),
                                                       (t.numpy() for t in _rank_grads(1, step)))]
        for i in range(len(SHAPES)):
            params[i], moms[i], _ = oracle.muon_matrix(params[i], g[i], moms[i], lr=np.float32(0.02),
                                                       beta=np.float32(0.95), nesterov=True, ns_steps=3)
    for i in range(len(SHAPES)):
        assert np.allclose(res[0][0][i], params[i], rtol=0, atol=1e-6), i
        assert np.allclose(res[owner[i]][2][i], moms[i], rtol=0, atol=1e-9), i


def _failing_worker(rank, world, port, case, out):
    import datetime
    import time
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=2))
    try:
        params = [workloads.make_param("zero2", i, s, "cpu", 0) for i, s in enumerate(SHAPES)]
        before = [p.clone() for p in params]

        def broken_compute(*args, **kwargs):
            raise RuntimeError("update failed on this rank")

        compute = broken_compute if (case == "raises" and rank == 1) else oracle_compute
        sharded = mu.zero2.ShardedMuon(params, compute=compute)
        if case == "never_joins" and rank == 1:
            time.sleep(6.0)  # holds the group open past the survivor's timeout, then leaves
            out[rank] = ("left", None, None)
            return
        t0 = time.monotonic()
        try:
            sharded.step(_rank_grads(rank, 0), **HYPER)
            out[rank] = ("ok", time.monotonic() - t0, None)
        except RuntimeError as e:
            # which matrices changed: a failure in phase 1 leaves every weight as it was
            changed = [i for i, (a, b) in enumerate(zip(before, params)) if not torch.equal(a, b)]
            out[rank] = (str(e)[:200], time.monotonic() - t0, (changed, sharded.owned))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", ["never_joins", "raises"])
def test_a_failed_rank_surfaces_as_an_error_on_the_others(case):
    world = 2
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_failing_worker, args=(world, _free_port(), case, out), nprocs=world, join=True)
        res = dict(out)
    msg, elapsed, state = res[0]
    assert msg != "ok", "the surviving rank finished a step its peer never completed"
    assert elapsed < 5.0  # the process group's 2 s limit ends the wait, not the peer's exit
    changed, owned = state
    if case == "never_joins":
        # the reduce-scatter never completed: no weight was touched
        assert changed == []
        assert res[1][0] == "left"
    else:
        # the peer failed after the reduce-scatter: only the survivor's own matrices moved
        assert set(changed) <= set(owned)
        assert "update failed" in res[1][0]
