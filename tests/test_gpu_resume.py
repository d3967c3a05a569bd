"""Checkpoint and resume of a training run's Muon steps (CUDA path, through the C ABI).

The library keeps no optimizer state of its own: the weights and the momentum
buffers belong to the caller, and the workspace is scratch rebuilt from the
shapes.  So a run that checkpoints its weights and momentum to host memory,
ends the context (muon_destroy), and resumes from the checkpoint into freshly
allocated tensors under a new context must continue exactly as a run that
never stopped: the training scripts the pages describe resume a pretraining
run from a saved step ("--resume-from-step"), and a resumed run must not
drift from an uninterrupted one.  The check is bitwise, over 20 carried steps
of the d26 stack with a fresh gradient draw every step.
"""
import pytest
import torch

import pretraining_optimizer_step_b300 as mu
import workloads

pytestmark = pytest.mark.gpu

HP = dict(lr=0.02, beta=0.95, nesterov=True, ns_steps=5)


def _steps(p, m, name, shapes, first, last):
    for step in range(first, last):
        g = [workloads.make_grad(name, i, s, "cuda", 0, step) for i, s in enumerate(shapes)]
        mu.muon_step(p, g, m, **HP)
        del g
    mu.muon_get_status()


@pytest.mark.slow
@pytest.mark.parametrize("name,steps", [("d2", 20), ("d26", 20)])
def test_resume_from_a_checkpoint_is_bitwise_equal_to_an_uninterrupted_run(name, steps):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    half = steps // 2
    # the uninterrupted run
    p, _, m, shapes = workloads.make_stack(name, "cuda")
    mu.muon_init(wait_timeout_s=2.0)
    try:
        _steps(p, m, name, shapes, 0, steps)
    finally:
        mu.muon_destroy()
    straight_p = [t.cpu() for t in p]
    straight_m = [t.cpu() for t in m]
    del p, m
    torch.cuda.empty_cache()

    # the interrupted run: checkpoint after `half` steps, end the context, drop every device tensor
    p, _, m, _ = workloads.make_stack(name, "cuda")
    mu.muon_init(wait_timeout_s=2.0)
    try:
        _steps(p, m, name, shapes, 0, half)
    finally:
        mu.muon_destroy()
    ckpt_p = [t.cpu() for t in p]
    ckpt_m = [t.cpu() for t in m]
    del p, m
    torch.cuda.empty_cache()
    # resume: new tensors (new device addresses), a new context, the remaining steps
    p = [t.cuda() for t in ckpt_p]
    m = [t.cuda() for t in ckpt_m]
    mu.muon_init(wait_timeout_s=2.0)
    try:
        _steps(p, m, name, shapes, half, steps)
    finally:
        mu.muon_destroy()
    for i in range(len(shapes)):
        assert torch.equal(p[i].cpu(), straight_p[i]), ("p", i)
        assert torch.equal(m[i].cpu(), straight_m[i]), ("m", i)
