"""The sharded step's driver on the GPU with one NCCL rank (one rank owns every
matrix; the collectives still run, in place, through NCCL).  Over two steps
with momentum carried, in two buckets, it must match the fp64 oracle at the
parity tolerances, and give bit for bit what one muon_step over all matrices
gives (bucketing changes which launch a matrix is in, not its arithmetic)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
import pretraining_optimizer_step_b300 as mu
import workloads
from gpu_util import check_matrix

pytestmark = pytest.mark.gpu

HP = dict(lr=0.02, beta=0.95, nesterov=True, ns_steps=5)


def test_single_rank_sharded_step_matches_the_oracle_and_muon_step():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    mu.muon_init(wait_timeout_s=2.0)
    try:
        p, g, m, shapes = workloads.make_stack("d2", "cuda")
        p_ref = [t.clone() for t in p]
        m_ref = [t.clone() for t in m]
        sharded = mu.zero2.ShardedMuon(p, buckets=2)
        assert len(sharded.buckets) == 2
        for i, t in sharded.momentum.items():
            t.copy_(m[i])
        for step in range(2):
            gs = g if step == 0 else [workloads.make_grad("d2", i, s, "cuda", 0, step) for i, s in enumerate(shapes)]
            p0 = [t.cpu().numpy() for t in p]
            g0 = [t.cpu().numpy() for t in gs]
            m0 = [sharded.momentum[i].cpu().numpy() for i in range(len(p))]
            sharded.step(gs, **HP)
            mu.muon_step(p_ref, gs, m_ref, **HP)
            mu.muon_get_status()
            torch.cuda.synchronize()
            for i in range(len(p)):
                check_matrix(i, p0[i], g0[i], m0[i], p[i].cpu().numpy(), sharded.momentum[i].cpu().numpy(), None,
                             HP["lr"], HP["beta"], True, HP["ns_steps"], oracle.DEFAULT_COEFFS)
                assert torch.equal(p[i], p_ref[i]), (step, i)
                assert torch.equal(sharded.momentum[i], m_ref[i]), (step, i)
    finally:
        mu.muon_destroy()
        dist.destroy_process_group()
