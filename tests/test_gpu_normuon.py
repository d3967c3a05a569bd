"""Parity of the CUDA Muon step with NorMuon scaling (muon_step_normuon, through
the C ABI) with the fp64 oracle on the same inputs.

Tolerances (per matrix, relative Frobenius): the scaled update O' within 2e-2
and the updated weights within 1e-3, as for muon_step; the second-moment state
V' within 2e-2 (its per-row means are taken of the bf16-computed update); the
momentum buffer within float32 rounding of its terms.  The context is the one a
caller makes (debug_flags = 0); O' is recovered from the weight change
(p' = p - lr sqrt(max(1, r/c)) O'), and the debug copy of O' has its own test.
"""
import numpy as np
import pytest
import torch

import oracle
import pretraining_optimizer_step_b300 as mu
import workloads
from gpu_util import TOL_O, TOL_P, TOL_DP, check_momentum, o_from_update, rel_fro

pytestmark = pytest.mark.gpu

BETA2 = 0.95
EPS2 = 1e-10


@pytest.fixture(autouse=True)
def fresh_context():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mu.muon_init(wait_timeout_s=2.0)
    yield
    mu.muon_destroy()


def cpu(ts):
    return [t.detach().cpu().numpy().copy() for t in ts]


def step_and_check(p, g, m, V, ns_steps=5, tol_o=TOL_O, check_idx=None, keep_o=False):
    """keep_o: the context keeps the debug copy of O', which is checked instead of the O'
    recovered from the weight change."""
    p0, g0, m0, V0 = cpu(p), cpu(g), cpu(m), cpu(V)
    mu.muon_step_normuon(p, g, m, V, lr=0.02, beta=0.95, nesterov=True, ns_steps=ns_steps, beta2=BETA2, eps2=EPS2)
    mu.muon_get_status()
    idx = range(len(p)) if check_idx is None else check_idx
    worst = {}
    for i in idx:
        p1 = p[i].cpu().numpy()
        if keep_o:
            O = torch.empty_like(p[i])
            mu.muon_debug_copy_ns_output(i, O)
            torch.cuda.synchronize()
            O = O.cpu().numpy()
        else:
            O = o_from_update(p0[i], p1, 0.02, p0[i].shape)
        p_ref, m_ref, V_ref, O_ref = oracle.normuon_matrix(p0[i], g0[i], m0[i], V0[i], lr=np.float32(0.02),
                                                           beta=np.float32(0.95), ns_steps=ns_steps,
                                                           beta2=np.float32(BETA2), eps2=np.float32(EPS2))
        rep = {"O": rel_fro(O, O_ref), "p": rel_fro(p1, p_ref),
               "dp": rel_fro(p1.astype(np.float64) - p0[i], p_ref.astype(np.float64) - p0[i]),
               "V": rel_fro(V[i].cpu().numpy(), V_ref)}
        assert rep["O"] <= tol_o and rep["p"] <= TOL_P and rep["dp"] <= TOL_DP and rep["V"] <= 2e-2, (i, rep)
        check_momentum(i, g0[i], m0[i], m[i].cpu().numpy(), m_ref, 0.95)
        for k, v in rep.items():
            worst[k] = max(worst.get(k, 0.0), v)
    return worst


def zeros_state(shapes):
    return [torch.zeros(r, device="cuda") for r, _ in shapes]


def test_d2_full_stack_from_zero_state():
    p, g, m, shapes = workloads.make_stack("d2", "cuda")
    step_and_check(p, g, m, zeros_state(shapes))


def test_two_steps_carry_the_state():
    name = "d2"
    p, g, m, shapes = workloads.make_stack(name, "cuda")
    V = zeros_state(shapes)
    step_and_check(p, g, m, V)
    g2 = [workloads.make_grad(name, i, s, "cuda", 0, 1) for i, s in enumerate(shapes)]
    step_and_check(p, g2, m, V)


def test_ragged_and_tall_wide_shapes():
    shapes = [(136, 200), (200, 136), (264, 264), (392, 1032), (1032, 392)]
    p, g, m, _ = workloads.make_custom(shapes, "cuda", tag="normuon")
    V = [torch.rand(r, device="cuda") * 1e-3 for r, _ in shapes]
    step_and_check(p, g, m, V)


def test_d12_sampled():
    p, g, m, shapes = workloads.make_stack("d12", "cuda")
    step_and_check(p, g, m, zeros_state(shapes), check_idx=[0, 4, 5, 70, 71])


@pytest.mark.slow
def test_d26_sampled():
    # the configuration the benchmark's NorMuon leg times (the full d26 stack, a zero state);
    # the oracle checks the first and last layers' square, tall and wide matrices
    p, g, m, shapes = workloads.make_stack("d26", "cuda")
    n = len(p)
    assert shapes[4] == (6656, 1664) and shapes[n - 1] == (1664, 6656)
    step_and_check(p, g, m, zeros_state(shapes), check_idx=[0, 4, 5, n - 6, n - 2, n - 1])


def test_zero_gradient_leaves_weights_and_decays_state():
    shapes = [(64, 64), (256, 64), (64, 256)]
    p = [torch.randn(s, device="cuda") for s in shapes]
    g = [torch.zeros(s, device="cuda") for s in shapes]
    m = [torch.zeros(s, device="cuda") for s in shapes]
    V = [torch.full((r,), 0.5, device="cuda") for r, _ in shapes]
    p0 = [t.clone() for t in p]
    mu.muon_step_normuon(p, g, m, V, beta2=BETA2, eps2=EPS2)
    mu.muon_get_status()
    for i in range(3):
        assert torch.equal(p[i], p0[i])
        assert torch.allclose(V[i], torch.full_like(V[i], np.float32(BETA2) * 0.5), rtol=1e-6, atol=0)


def test_argument_errors():
    p, g, m, shapes = workloads.make_custom([(64, 64), (64, 128)], "cuda", tag="nmargs")
    V = zeros_state(shapes)
    before = [t.clone() for t in p + m + V]
    assert mu.muon_step_normuon(p, g, m, V, ns_steps=0, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_step_normuon(p, g, m, V, beta2=1.0, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_step_normuon(p, g, m, [V[0].data_ptr() + 2, V[1]], check=False) == mu.MUON_ERR_MISALIGNED
    assert mu.muon_step_normuon(p, g, m, [V[0], 0], check=False) == mu.MUON_ERR_INVALID_ARG
    torch.cuda.synchronize()
    for a, b in zip(before, p + m + V):
        assert torch.equal(a, b)


@pytest.mark.parametrize("case", ["d2", "ragged"])
def test_row_statistics_are_consistent_with_the_update(case):
    # With a zero state, V'_i = (1 - beta2) mean_j O_ij^2, and the applied update is O' = step_i ratio O
    # with step_i = 1 / sqrt(V'_i + eps2).  So every stored row gives the same value
    #   mean_j O'_ij^2 (V'_i + eps2) (1 - beta2) / V'_i  =  ratio^2,
    # to float32 rounding (and the recovery of O' from p').  A row sum that missed or double-counted part of its row (a tile, a
    # ragged edge, a 32-row group of a transposed matrix) breaks the equality for that row.
    if case == "d2":
        p, g, m, shapes = workloads.make_stack("d2", "cuda")
    else:
        shapes = [(136, 200), (200, 136), (264, 264), (392, 1032), (1032, 392), (8, 1024), (1024, 8)]
        p, g, m, _ = workloads.make_custom(shapes, "cuda", tag="nmrows")
    V = zeros_state(shapes)
    p0 = cpu(p)
    mu.muon_step_normuon(p, g, m, V, lr=0.02, beta=0.95, nesterov=True, ns_steps=5, beta2=BETA2, eps2=EPS2)
    mu.muon_get_status()
    for i, (r, c) in enumerate(shapes):
        # O' from the weight change: float32 rounding of p' costs at most a few 1e-6 of each entry
        Op = o_from_update(p0[i], p[i].cpu().numpy(), 0.02, (r, c))
        Vi = V[i].double().cpu().numpy()
        assert np.all(Vi > 0), i
        r2 = np.mean(Op * Op, axis=1) * (Vi + EPS2) * (1.0 - float(np.float32(BETA2))) / Vi
        assert np.max(np.abs(r2 / np.median(r2) - 1.0)) <= 1e-4, (i, float(np.max(np.abs(r2 / np.median(r2) - 1.0))))


@pytest.mark.parametrize("ns_steps,tol", [(1, 5e-3), (2, TOL_O)])
def test_short_iterations_on_ragged_shapes(ns_steps, tol):
    # with one iteration the launch that writes O is also the first one, so it applies the
    # 1/||u|| scale itself; the single iteration is checked tightly (bf16 rounding of X0 gives
    # about 1.7e-3), as for muon_step
    shapes = [(136, 200), (200, 136), (264, 264), (8, 1024), (1024, 8)]
    p, g, m, _ = workloads.make_custom(shapes, "cuda", tag="nmshort")
    V = [torch.rand(r, device="cuda") * 1e-3 for r, _ in shapes]
    step_and_check(p, g, m, V, ns_steps=ns_steps, tol_o=tol)


def test_debug_copy_of_the_scaled_update():
    # MUON_DEBUG_KEEP_O makes the update kernel also store O' = step_i ratio O; it must match the
    # oracle, and the step must leave weights, momentum and state bit for bit as without it
    shapes = [(136, 200), (200, 136), (264, 264), (8, 1024), (1024, 8)]
    p, g, m, _ = workloads.make_custom(shapes, "cuda", tag="nmdbg")
    V = [torch.rand(r, device="cuda") * 1e-3 for r, _ in shapes]
    snap = [t.clone() for t in p + g + m + V]
    mu.muon_step_normuon(p, g, m, V, lr=0.02, beta=0.95, nesterov=True, ns_steps=5, beta2=BETA2, eps2=EPS2)
    mu.muon_get_status()
    plain = [t.clone() for t in p + m + V]
    mu.muon_destroy()
    mu.muon_init(debug_flags=mu.MUON_DEBUG_KEEP_O, wait_timeout_s=2.0)
    for dst, src in zip(p + g + m + V, snap):
        dst.copy_(src)
    step_and_check(p, g, m, V, keep_o=True)
    for a, b in zip(plain, p + m + V):
        assert torch.equal(a, b)
