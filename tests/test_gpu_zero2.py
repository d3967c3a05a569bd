"""The sharded step's driver on the GPU with one NCCL rank: it must reproduce
muon_step bitwise (one rank owns every matrix; the collectives copy)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist

import pretraining_optimizer_step_b300 as mu
import workloads

pytestmark = pytest.mark.gpu


def test_single_rank_sharded_step_equals_muon_step():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    mu.muon_init()
    try:
        p, g, m, shapes = workloads.make_stack("d2", "cuda")
        p_ref = [t.clone() for t in p]
        m_ref = [t.clone() for t in m]
        sharded = mu.zero2.ShardedMuon(p, stream=torch.cuda.current_stream())
        for i, t in sharded.momentum.items():
            t.copy_(m[i])
        for step in range(2):
            gs = g if step == 0 else [workloads.make_grad("d2", i, s, "cuda", 0, step) for i, s in enumerate(shapes)]
            sharded.step(gs, lr=0.02, beta=0.95, nesterov=True, ns_steps=5)
            mu.muon_step(p_ref, gs, m_ref, lr=0.02, beta=0.95, nesterov=True, ns_steps=5)
        mu.muon_get_status()
        torch.cuda.synchronize()
        for i in range(len(p)):
            assert torch.equal(p[i], p_ref[i]), i
            assert torch.equal(sharded.momentum[i], m_ref[i]), i
    finally:
        mu.muon_destroy()
        dist.destroy_process_group()
