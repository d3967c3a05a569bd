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


def _worker(rank, world, port, buckets, zero_copy, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        params = [workloads.make_param("zero2", i, s, "cpu", 0) for i, s in enumerate(SHAPES)]
        ids = [id(p) for p in params]
        sharded = mu.zero2.ShardedMuon(params, compute=oracle_compute, buckets=buckets)
        # the caller's tensors are the same objects, now living in the bucket buffers
        assert [id(p) for p in params] == ids
        assert all(torch.equal(p, workloads.make_param("zero2", i, s, "cpu", 0))
                   for i, (p, s) in enumerate(zip(params, SHAPES)))
        for step in range(2):
            if zero_copy:
                for i, g in enumerate(_rank_grads(rank, step)):
                    sharded.grad_view(i).copy_(g)
                sharded.step(**HYPER)
            else:
                sharded.step(_rank_grads(rank, step), **HYPER)
        out[rank] = ([p.numpy().copy() for p in params], sharded.owner,
                     {i: m.numpy().copy() for i, m in sharded.momentum.items()}, len(sharded.buckets))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,buckets,zero_copy", [(2, 1, False), (2, 2, False), (3, 3, True), (3, 2, False)])
def test_gloo_ranks_match_one_process_on_the_mean_gradient(world, buckets, zero_copy):
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), buckets, zero_copy, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][3] == buckets
    # every rank ends with the same weights
    for r in range(1, world):
        for a, b in zip(res[0][0], res[r][0]):
            assert np.array_equal(a, b)
    owner = res[0][1]
    assert sorted(set(owner)) == list(range(world))
    # reference: one process, the mean of the ranks' gradients, full momentum (the oracle)
    params = [workloads.make_param("zero2", i, s, "cpu", 0).numpy() for i, s in enumerate(SHAPES)]
    moms = [np.zeros(s, np.float32) for s in SHAPES]
    for step in range(2):
        per_rank = [[t.numpy() for t in _rank_grads(r, step)] for r in range(world)]
        g = [(sum(gs[i].astype(np.float64) for gs in per_rank) / world).astype(np.float32) for i in range(len(SHAPES))]
        for i in range(len(SHAPES)):
            params[i], moms[i], _ = oracle.muon_matrix(params[i], g[i], moms[i], lr=np.float32(0.02),
                                                       beta=np.float32(0.95), nesterov=True, ns_steps=3)
    for i in range(len(SHAPES)):
        assert np.allclose(res[0][0][i], params[i], rtol=0, atol=1e-6), i
        assert np.allclose(res[owner[i]][2][i], moms[i], rtol=0, atol=1e-9), i


def test_buckets_cut_at_about_equal_sizes():
    # host logic of the split, through a one-rank gloo group: consecutive matrices in index
    # order, every matrix in exactly one bucket, at most the requested count, sizes within one
    # matrix of the mean
    params = [torch.zeros(s) for s in workloads.config_shapes("d2")]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        for nb in (1, 2, 3, 12, 20):
            sh = mu.zero2.ShardedMuon([p.clone() for p in params], compute=oracle_compute, buckets=nb)
            idx = [i for bk in sh.buckets for i in bk.index]
            assert idx == list(range(len(params)))
            assert 1 <= len(sh.buckets) <= min(nb, len(params)) and all(bk.index for bk in sh.buckets)
            if nb <= 3:
                assert len(sh.buckets) == nb
            sizes = [sum(params[i].numel() for i in bk.index) for bk in sh.buckets]
            assert max(sizes) <= sum(sizes) / len(sizes) + max(p.numel() for p in params)
    finally:
        dist.destroy_process_group()


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
        sharded = mu.zero2.ShardedMuon(params, compute=compute, buckets=2)
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
