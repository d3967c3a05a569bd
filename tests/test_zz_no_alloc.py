"""The allocation-free momentum + norm entry point, against muon_step and the oracle.

muon_momentum_norm_noalloc serves callers that cannot allocate device memory:
a process whose memory another runtime's pool already owns, or a service that
must not call cudaMalloc/cudaFree (both may synchronise the device) once it is
running.  It runs the same momentum + norm kernel as muon_step, with its
scratch in a fixed array inside the library instead of muon_step's workspace.

The checks, each over two calls in a row (momentum carried, a fresh gradient
for the second call):
  * against the existing entry point: the momentum buffer muon_step writes (bit
    for bit: same kernel, same arithmetic), the norms it records, and a bf16
    direction that, divided by (||u|| + eps), gives the O that muon_step applies
    at ns_steps = 0 (recovered from its weight change, tests/gpu_util.py);
  * against the oracle: m' within float32 rounding of its terms, ||u||_F within
    1e-5, and every entry of the direction within one bf16 rounding (relative
    2^-8) of the oracle's u;
  * the chunked path: more than 192 matrices (several launches sharing the
    scratch partials, tickets cleared once for all of them);
  * a request beyond the fixed scratch is refused before any work is enqueued.
This file is collected last, so a run that stops at its first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import pretraining_optimizer_step_b300 as mu
import workloads
from gpu_util import check_momentum, o_from_update, rel_fro, update_scale

pytestmark = pytest.mark.gpu

EPS = 1e-7
BETA = 0.95
BF16_REL = 2.0 ** -8   # round to nearest, 8 significant bits: |bf16(x) - x| <= 2^-8 |x|


def _oriented_back(x0, shape):
    r, c = shape
    x = x0.float().cpu().numpy().astype(np.float64)
    return x.reshape(c, r).T if r > c else x.reshape(r, c)


def _check_against_oracle(i, g0, m0, m1, x0, norm):
    m_ref, u = oracle.momentum(g0, m0, np.float32(BETA), True)
    check_momentum(i, g0, m0, m1, m_ref, BETA)
    nrm = float(np.linalg.norm(u))
    assert abs(norm - nrm) <= 1e-5 * nrm, (i, norm, nrm)
    # the GPU forms u in fp32 with two fmas (m' = beta m + g, u = g + beta m'), within a few
    # float32 ulps of the terms, then rounds it to bf16 once
    g64, m64 = g0.astype(np.float64), m0.astype(np.float64)
    terms = np.abs(g64) + BETA * (BETA * np.abs(m64) + np.abs(g64))
    assert np.all(np.abs(x0 - u) <= BF16_REL * np.abs(u) + 4e-7 * terms), i


def _run_two_calls(name, shapes, p, g, m, check_oracle_idx):
    m_na = [t.clone() for t in m]
    x0 = [torch.empty(r * c, dtype=torch.bfloat16, device="cuda") for r, c in shapes]
    norms = torch.empty(len(shapes), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    for call in range(2):
        if call > 0:
            g = [workloads.make_grad(name, i, s, "cuda", 0, call) for i, s in enumerate(shapes)]
        g0 = {i: g[i].cpu().numpy() for i in check_oracle_idx}
        m0 = {i: m_na[i].cpu().numpy() for i in check_oracle_idx}
        p0 = [t.cpu().numpy() for t in p]
        # existing entry point: momentum + norm, then p -= lr s X0 / (||u|| + eps)
        mu.muon_step(p, g, m, lr=0.02, beta=BETA, nesterov=True, ns_steps=0, stream=stream)
        mu.muon_get_status(stream)
        norms_ref = mu.muon_debug_copy_norms(len(shapes))
        # the allocation-free entry point on the same gradient
        for t in x0:
            t.fill_(float("nan"))
        norms.fill_(float("nan"))
        mu.muon_momentum_norm_noalloc(g, m_na, x0, norms, beta=BETA, nesterov=True, stream=stream)
        torch.cuda.synchronize()

        got_norms = norms.cpu().numpy()
        for i, s in enumerate(shapes):
            # same kernel and arithmetic: the momentum buffers agree exactly
            assert torch.equal(m_na[i], m[i]), (call, i)
            ref = norms_ref[i]
            assert abs(got_norms[i] - ref) <= 1e-6 * ref, (call, i, got_norms[i], ref)
            x = _oriented_back(x0[i], s)
            O_na = x / (float(got_norms[i]) + EPS)
            p1 = p[i].cpu().numpy()
            O_step = o_from_update(p0[i], p1, 0.02, s)
            # O recovered from p' = p - sc O carries p''s float32 rounding (at most 2^-24 |p'| per
            # entry) divided by sc; at ns_steps = 0, ||O||_F is 1, so that is a few 1e-5 here
            bound = 2.0 ** -23 * np.linalg.norm(p1) / (float(update_scale(0.02, s)) * np.linalg.norm(O_step)) + 1e-6
            err = rel_fro(O_na, O_step)
            assert err <= bound, (call, i, err, bound)
            if i in check_oracle_idx:
                _check_against_oracle(i, g0[i], m0[i], m_na[i].cpu().numpy(), x, float(got_norms[i]))


@pytest.fixture
def context():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mu.muon_init(wait_timeout_s=2.0)
    yield
    mu.muon_destroy()


def test_noalloc_matches_muon_step_and_the_oracle_on_two_calls_in_a_row(context):
    name = "d2"
    p, g, m, shapes = workloads.make_stack(name, "cuda")
    _run_two_calls(name, shapes, p, g, m, check_oracle_idx=list(range(len(shapes))))


def test_noalloc_more_than_192_matrices_take_several_launches(context):
    # 260 matrices (two launches of at most 192): squares, 4:1 tall (transposed) and wide,
    # and ragged shapes, so both launches hold every kind; the oracle checks matrices from both
    base = [(256, 256), (512, 128), (128, 512), (136, 200), (200, 136)]
    shapes = [base[i % len(base)] for i in range(260)]
    p, g, m, _ = workloads.make_custom(shapes, "cuda", tag="noalloc260")
    _run_two_calls("noalloc260", shapes, p, g, m, check_oracle_idx=[0, 1, 2, 3, 4, 190, 191, 192, 193, 259])


def test_noalloc_refuses_requests_beyond_its_scratch():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    # 1025 matrices: one more than the fixed scratch holds tickets for
    shapes = [(8, 8)] * 1025
    g = [torch.randn(8, 8, device="cuda") for _ in shapes]
    m = [torch.randn(8, 8, device="cuda") for _ in shapes]
    x0 = [torch.zeros(64, dtype=torch.bfloat16, device="cuda") for _ in shapes]
    norms = torch.full((len(shapes),), -1.0, device="cuda")
    before = [t.clone() for t in m]
    st = mu.muon_momentum_norm_noalloc(g, m, x0, norms, check=False)
    assert st == mu.MUON_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    for a, b in zip(before, m):
        assert torch.equal(a, b)
    assert bool((norms == -1.0).all())
    assert all(int(torch.count_nonzero(t.float())) == 0 for t in x0)
    # the same request within the limit then runs
    assert mu.muon_momentum_norm_noalloc(g[:1024], m[:1024], x0[:1024], norms, check=False) == mu.MUON_OK
    torch.cuda.synchronize()
    assert bool((norms[:1024] > 0).all())
