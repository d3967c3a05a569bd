"""The allocation-free momentum + norm entry point against muon_step's own pass.

muon_momentum_norm_noalloc serves callers that cannot allocate device memory:
a process whose memory another runtime's pool already owns, or a service that
must not call cudaMalloc/cudaFree (both may synchronise the device) once it is
running.  It runs the same momentum + norm kernel as muon_step, with its
scratch in a fixed array inside the library instead of muon_step's workspace.

The check: over two calls in a row (momentum carried, a fresh gradient for the
second call), it must give the momentum buffer muon_step writes, the norms
muon_step records, and a bf16 direction that, divided by (||u|| + eps), equals
muon_step's O at ns_steps = 0.  The tolerances are the ones the parity tests
use (tests/gpu_util.py).  This file is collected last, so a run that stops at
its first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import pretraining_optimizer_step_b300 as mu
import workloads
from gpu_util import TOL_O, rel_fro

pytestmark = pytest.mark.gpu

EPS = 1e-7


def _oriented_back(x0, shape):
    r, c = shape
    x = x0.float().cpu().numpy().astype(np.float64)
    return x.reshape(c, r).T if r > c else x.reshape(r, c)


def test_noalloc_matches_muon_step_on_two_calls_in_a_row():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    name = "d2"
    p, g, m, shapes = workloads.make_stack(name, "cuda")
    # the no-alloc side works on its own copy of the momentum
    m_na = [t.clone() for t in m]
    x0 = [torch.empty(r * c, dtype=torch.bfloat16, device="cuda") for r, c in shapes]
    norms = torch.empty(len(shapes), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    mu.muon_init(debug_flags=mu.MUON_DEBUG_KEEP_O, wait_timeout_s=2.0)
    try:
        for call in range(2):
            if call > 0:
                g = [workloads.make_grad(name, i, s, "cuda", 0, call) for i, s in enumerate(shapes)]
            # existing entry point: momentum + norm, then O = X0 / (||u|| + eps)
            mu.muon_step(p, g, m, lr=0.02, beta=0.95, nesterov=True, ns_steps=0, stream=stream)
            mu.muon_get_status(stream)
            O_ref = []
            for i, t in enumerate(p):
                o = torch.empty_like(t)
                mu.muon_debug_copy_ns_output(i, o, stream)
                O_ref.append(o)
            norms_ref = mu.muon_debug_copy_norms(len(shapes))
            # the allocation-free entry point on the same gradient
            for t in x0:
                t.fill_(float("nan"))
            mu.muon_momentum_norm_noalloc(g, m_na, x0, norms, beta=0.95, nesterov=True, stream=stream)
            torch.cuda.synchronize()

            got_norms = norms.cpu().numpy()
            for i, s in enumerate(shapes):
                # same kernel and arithmetic: the momentum buffers agree exactly
                assert torch.equal(m_na[i], m[i]), (call, i)
                ref = norms_ref[i]
                assert abs(got_norms[i] - ref) <= 1e-5 * ref, (call, i, got_norms[i], ref)
                O_na = _oriented_back(x0[i], s) / (float(got_norms[i]) + EPS)
                err = rel_fro(O_na, O_ref[i].cpu().numpy())
                assert err <= TOL_O, (call, i, err)
    finally:
        mu.muon_destroy()
