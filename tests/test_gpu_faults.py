"""Failure detection on the GPU without a GPU fault.

Every in-kernel wait of the library is bounded (poll count and wall clock).
The test hook MUON_DEBUG_INJECT_LOST_LOAD makes the even CTA of the first pair
of the first Gram launch skip one operand panel, so that stage's barrier never
completes: the MMA issuer's wait must expire, every role of the pair must stop
within its own limit, the step must report MUON_ERR_DEVICE_TIMEOUT through
muon_get_status, and the context must stay usable for the next step.
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
