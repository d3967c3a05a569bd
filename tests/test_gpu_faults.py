"""Failure detection on the GPU without a GPU fault.

Every in-kernel wait of the library is bounded (poll count and wall clock).
The test hook MUON_DEBUG_INJECT_LOST_LOAD makes the even CTA of the first pair
of the first Gram launch skip one operand panel, so that stage's barrier never
completes: the MMA issuer's wait must expire, every role of the pair must stop
within its own limit, the step must report MUON_ERR_DEVICE_TIMEOUT through
muon_get_status, and the context must stay usable for the next step.
MUON_DEBUG_INJECT_BAD_TILES gives a launch a tile list that does not match its
classes: the kernel must refuse it (MUON_ERR_DEVICE_BOUNDS).  A workspace
request beyond the device's memory must fail with MUON_ERR_OUT_OF_MEMORY
before anything is enqueued.
"""
import numpy as np
import pytest
import torch

import pretraining_optimizer_step_b300 as mu
import workloads
from gpu_util import TOL_O, check_matrix, run_gpu_step
import oracle

pytestmark = pytest.mark.gpu


def test_lost_load_times_out_and_the_context_survives():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mu.muon_init(debug_flags=mu.MUON_DEBUG_INJECT_LOST_LOAD, wait_timeout_s=0.2)
    try:
        p, g, m, _ = workloads.make_stack("d2", "cuda")
        mu.muon_step(p, g, m)
        assert mu.muon_get_status(check=False) == mu.MUON_ERR_DEVICE_TIMEOUT
        # the status word is cleared once read
        assert mu.muon_get_status(check=False) == mu.MUON_OK
    finally:
        mu.muon_destroy()
    # a fresh context on the same device computes a correct step
    mu.muon_init(wait_timeout_s=2.0)
    try:
        p, g, m, _ = workloads.make_stack("d2", "cuda")
        p0, g0, m0 = ([t.cpu().numpy().copy() for t in ts] for ts in (p, g, m))
        run_gpu_step(p, g, m)
        for i in (0, 4, 5):
            check_matrix(i, p0[i], g0[i], m0[i], p[i].cpu().numpy(), m[i].cpu().numpy(), None, 0.02, 0.95, True, 5,
                         oracle.DEFAULT_COEFFS)
    finally:
        mu.muon_destroy()


def test_inconsistent_tile_list_is_refused_with_a_bounds_status():
    # MUON_DEBUG_INJECT_BAD_TILES gives the first Gram launch one tile more than its classes hold;
    # every CTA of that launch must see the mismatch, run no tile, and latch the bounds status,
    # which muon_get_status turns into MUON_ERR_DEVICE_BOUNDS.  No wait times out (no hang), and
    # the context computes a correct step afterwards
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mu.muon_init(debug_flags=mu.MUON_DEBUG_INJECT_BAD_TILES, wait_timeout_s=2.0)
    try:
        p, g, m, _ = workloads.make_stack("d2", "cuda")
        import time
        t0 = time.monotonic()
        mu.muon_step(p, g, m)
        assert mu.muon_get_status(check=False) == mu.MUON_ERR_DEVICE_BOUNDS
        assert time.monotonic() - t0 < 1.5  # refused at once, not after a wait limit
        assert mu.muon_get_status(check=False) == mu.MUON_OK
        # the hook fires once per context: the next step is whole again
        p, g, m, _ = workloads.make_stack("d2", "cuda")
        p0, g0, m0 = ([t.cpu().numpy().copy() for t in ts] for ts in (p, g, m))
        run_gpu_step(p, g, m)
        for i in (0, 4, 5):
            check_matrix(i, p0[i], g0[i], m0[i], p[i].cpu().numpy(), m[i].cpu().numpy(), None, 0.02, 0.95, True, 5,
                         oracle.DEFAULT_COEFFS)
    finally:
        mu.muon_destroy()


def test_workspace_allocation_failure_is_reported_and_enqueues_nothing():
    # ten 65536 x 65536 matrices need about 344 GB of workspace, more than the device holds: the
    # step must return MUON_ERR_OUT_OF_MEMORY from the workspace allocation, before anything is
    # enqueued (the weight, gradient and momentum pointers are never touched, so aligned stand-in
    # addresses serve), and the context must still run a correct step
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mu.muon_init(wait_timeout_s=2.0)
    try:
        n = 10
        shapes = [(65536, 65536)] * n
        fake = [(1 << 40) + 4096 * i for i in range(n)]
        args = mu.StepArgs(fake, fake, fake, shapes=shapes)
        assert mu.muon_step(args, check=False) == mu.MUON_ERR_OUT_OF_MEMORY
        torch.cuda.synchronize()
        assert mu.muon_get_status(check=False) == mu.MUON_OK
        p, g, m, _ = workloads.make_stack("d2", "cuda")
        p0, g0, m0 = ([t.cpu().numpy().copy() for t in ts] for ts in (p, g, m))
        run_gpu_step(p, g, m)
        for i in (0, 4, 5):
            check_matrix(i, p0[i], g0[i], m0[i], p[i].cpu().numpy(), m[i].cpu().numpy(), None, 0.02, 0.95, True, 5,
                         oracle.DEFAULT_COEFFS)
    finally:
        mu.muon_destroy()
