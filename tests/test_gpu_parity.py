"""Parity of the CUDA Muon step (through the C ABI) with the fp64 oracle.

Every case draws seeded inputs from workloads.py on the device, keeps a CPU copy
of them, runs one muon_step, and compares each checked matrix with the oracle
run on the same CPU copy (tolerances in tests/gpu_util.py).  The context is the
one a caller makes (debug_flags = 0), so the launches checked are the ones the
benchmark times; O is recovered from the weight change.  The debug copy of O
(MUON_DEBUG_KEEP_O) has its own test, which also checks that it leaves the
weights bit for bit as the plain step does.
"""
import numpy as np
import pytest
import torch

import oracle
import pretraining_optimizer_step_b300 as mu
import workloads
from gpu_util import TOL_O, check_matrix, rel_fro, run_gpu_step

pytestmark = pytest.mark.gpu

DEFAULT = oracle.DEFAULT_COEFFS


@pytest.fixture(autouse=True)
def fresh_context():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mu.muon_init(wait_timeout_s=2.0)
    yield
    mu.muon_destroy()


def cpu_copy(ts):
    return [t.detach().cpu().numpy().copy() for t in ts]


def run_and_check(params, grads, moms, check_idx=None, lr=0.02, beta=0.95, nesterov=True, ns_steps=5,
                  coeffs=DEFAULT, mode=0, tol_o=None, keep_o=False):
    """tol_o: None (2e-2), a number, or a function of the stored shape.  keep_o: the context
    keeps the debug copy of O, which is checked instead of the O recovered from the update."""
    p0, g0, m0 = cpu_copy(params), cpu_copy(grads), cpu_copy(moms)
    O = run_gpu_step(params, grads, moms, lr=lr, beta=beta, nesterov=nesterov, ns_steps=ns_steps,
                     keep_o=keep_o)
    norms = mu.muon_debug_copy_norms(len(params))
    p1, m1 = cpu_copy(params), cpu_copy(moms)
    idx = range(len(params)) if check_idx is None else check_idx
    worst = {}
    for i in idx:
        tol = TOL_O if tol_o is None else (tol_o(p0[i].shape) if callable(tol_o) else tol_o)
        rep, _ = check_matrix(i, p0[i], g0[i], m0[i], p1[i], m1[i], O[i] if keep_o else None, lr, beta,
                              nesterov, ns_steps,
                              coeffs, mode=mode, norm_gpu=norms[i], tol_o=tol)
        for k, v in rep.items():
            worst[k] = max(worst.get(k, 0.0), v)
    return worst


def test_d2_full_stack():
    p, g, m, _ = workloads.make_stack("d2", "cuda")
    worst = run_and_check(p, g, m)
    assert worst["O"] < TOL_O


@pytest.mark.parametrize("ns_steps", [0, 1, 2])
def test_d2_short_iterations(ns_steps):
    p, g, m, _ = workloads.make_stack("d2", "cuda")
    run_and_check(p, g, m, ns_steps=ns_steps)


RAGGED = [(136, 200), (200, 136), (8, 8), (8, 1024), (1024, 8), (264, 264), (128, 384), (384, 128),
          (520, 64), (392, 1032), (1032, 392), (520, 1040), (1040, 520)]


def small_side_tol(shape):
    # below 64 rows or columns the Frobenius error of bf16 arithmetic does not
    # average out: over 40 seeded 8 x 8 inputs, a model of the kernels' rounding
    # points gives O errors up to 3.9e-2 against the fp64 oracle (median 1.4e-2);
    # tests/test_rounding_model.py runs that model on the CPU
    return TOL_O if min(shape) >= 64 else 6e-2


def pe_small_side_tol(shape):
    # with the Polar Express table, sides below 64 reach 8e-2 to 9e-2 in the rounding model (the
    # rows' large a I and b A terms cancel on bf16 operands); tests/test_rounding_model.py
    return TOL_O if min(shape) >= 64 else 1.2e-1


@pytest.mark.parametrize("ns_steps,tol", [(1, 5e-3), (5, small_side_tol)])
def test_ragged_and_edge_shapes(ns_steps, tol):
    # one iteration is checked tightly (bf16 rounding of X0 gives about 1.7e-3),
    # so any tile, mask or transpose error shows as an O(1) mismatch
    p, g, m, _ = workloads.make_custom(RAGGED, "cuda", tag="ragged")
    run_and_check(p, g, m, ns_steps=ns_steps, tol_o=tol)


@pytest.mark.parametrize("nesterov,mode", [(False, 0), (True, 1), (False, 1)])
def test_momentum_variants(nesterov, mode):
    mu.muon_destroy()
    mu.muon_init(momentum_mode=mode, wait_timeout_s=2.0)
    p, g, m, _ = workloads.make_stack("d2", "cuda")
    run_and_check(p, g, m, nesterov=nesterov, beta=0.9, lr=0.05, mode=mode)


def test_pages_polar_express_rows():
    # the two rows the pages print (3 decimals), each used for one iteration.
    # Only these two: the pages elide the other three, and following them with
    # the default row diverges (the composite scalar map passes 1e30 on parts
    # of (0, 1]), so a longer table of that mix has no meaningful result
    rows = [tuple(r) for r in oracle.PAGES_POLAR_EXPRESS_ROWS]
    mu.muon_destroy()
    mu.muon_init(coeffs=rows, wait_timeout_s=2.0)
    p, g, m, _ = workloads.make_stack("d2", "cuda")
    run_and_check(p, g, m, coeffs=np.array(rows), ns_steps=2)


@pytest.mark.parametrize("case", ["d2", "ragged"])
def test_derived_polar_express_table(case):
    # the full five-row table of the Polar Express construction (the two rows the pages print
    # and the three derived ones; tests/test_polar_express.py pins it on the CPU).  A model of
    # the kernels' rounding gives O errors of 1.3e-2 to 1.4e-2 with it on sides of 64 and more
    rows = [tuple(r) for r in mu.POLAR_EXPRESS_COEFFS]
    mu.muon_destroy()
    mu.muon_init(coeffs=rows, wait_timeout_s=2.0)
    if case == "d2":
        p, g, m, _ = workloads.make_stack("d2", "cuda")
    else:
        p, g, m, _ = workloads.make_custom(RAGGED, "cuda", tag="ragged")
    run_and_check(p, g, m, coeffs=np.array(rows), ns_steps=5, tol_o=pe_small_side_tol)


def test_per_iteration_rows_switch():
    # five iterations whose rows alternate between the default quintic and the
    # cubic Newton-Schulz step X <- 1.5 X - 0.5 X X^T X (a, b, c = 1.5, -0.5, 0):
    # a convergent table (outputs stay in (0, 1] on (0.001, 1]) in which every
    # launch must pick up its own row
    cubic = (1.5, -0.5, 0.0)
    rows = [oracle.DEFAULT_ROW, cubic, oracle.DEFAULT_ROW, cubic, cubic]
    mu.muon_destroy()
    mu.muon_init(coeffs=rows, wait_timeout_s=2.0)
    p, g, m, _ = workloads.make_stack("d2", "cuda")
    run_and_check(p, g, m, coeffs=np.array(rows), ns_steps=5)


def test_d12_stack_sampled():
    p, g, m, _ = workloads.make_stack("d12", "cuda")
    run_and_check(p, g, m, check_idx=[0, 3, 4, 5, 64, 70, 71])


def test_zero_gradient_and_momentum():
    shapes = [(64, 64), (256, 64), (64, 256)]
    p = [torch.randn(s, device="cuda") for s in shapes]
    g = [torch.zeros(s, device="cuda") for s in shapes]
    m = [torch.zeros(s, device="cuda") for s in shapes]
    p0 = [t.clone() for t in p]
    run_gpu_step(p, g, m)
    for i in range(3):
        assert torch.equal(p[i], p0[i])
        assert torch.count_nonzero(m[i]) == 0


def test_deterministic_and_poisoned_workspace_agree():
    p, g, m, _ = workloads.make_stack("d2", "cuda")
    snap = [t.clone() for t in p + g + m]
    run_gpu_step(p, g, m)
    first = [t.clone() for t in p + m]
    # same inputs again, with the bf16 workspace filled with NaN first
    mu.muon_destroy()
    mu.muon_init(debug_flags=mu.MUON_DEBUG_POISON_WORKSPACE, wait_timeout_s=2.0)
    n = len(p)
    for dst, src in zip(p + g + m, snap):
        dst.copy_(src)
    run_gpu_step(p, g, m)
    for a, b in zip(first, p + m):
        assert torch.equal(a, b)


def test_multi_step_momentum_carried():
    name = "d2"
    p, g, m, shapes = workloads.make_stack(name, "cuda")
    # the oracle carries its own weights and momentum from step to step
    p_ref, m_ref = cpu_copy(p), cpu_copy(m)
    for step in range(3):
        if step > 0:
            g = [workloads.make_grad(name, i, s, "cuda", 0, step) for i, s in enumerate(shapes)]
        g0 = cpu_copy(g)
        run_gpu_step(p, g, m)
        p1, m1 = cpu_copy(p), cpu_copy(m)
        for i in range(len(p)):
            p_ref[i], m_ref[i], _ = oracle.muon_matrix(p_ref[i], g0[i], m_ref[i], lr=np.float32(0.02),
                                                       beta=np.float32(0.95), nesterov=True, ns_steps=5)
            assert rel_fro(p1[i], p_ref[i]) <= 1e-3, (step, i)
            assert rel_fro(m1[i], m_ref[i]) <= 1e-6, (step, i)


def test_shape_list_changes_rebuild_the_plan():
    for name in ("d2", "ragged", "d2"):
        if name == "ragged":
            p, g, m, _ = workloads.make_custom(RAGGED[:4], "cuda", tag="ragged")
        else:
            p, g, m, _ = workloads.make_stack(name, "cuda")
        run_and_check(p, g, m, check_idx=[0, 1, 2, 3], tol_o=small_side_tol)


def test_argument_errors_enqueue_nothing():
    p, g, m, shapes = workloads.make_custom([(64, 64), (64, 128)], "cuda", tag="args")
    before = [t.clone() for t in p + m]
    # misaligned pointer (4 bytes into a buffer)
    args = mu.StepArgs([p[0].data_ptr() + 4, p[1]], g, m, shapes=shapes)
    assert mu.muon_step(args, check=False) == mu.MUON_ERR_MISALIGNED
    assert mu.muon_step(p, g, m, shapes=[(64, 64), (64, 132)], check=False) == mu.MUON_ERR_UNSUPPORTED_SHAPE
    assert mu.muon_step(p, g, m, ns_steps=6, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_step(p, g, m, ns_steps=-1, check=False) == mu.MUON_ERR_INVALID_ARG
    args = mu.StepArgs([p[0], 0], g, m, shapes=shapes)
    assert mu.muon_step(args, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_step([], [], [], check=False) == mu.MUON_OK
    torch.cuda.synchronize()
    for a, b in zip(before, p + m):
        assert torch.equal(a, b)
    assert mu.muon_get_status() == mu.MUON_OK


def test_step_info_counts_launches():
    p, g, m, shapes = workloads.make_stack("d2", "cuda")
    run_gpu_step(p, g, m)
    info = mu.muon_get_step_info()
    q = mu.muon_plan_query(shapes, 5)
    assert info["launches"] == q["launches"] == 16
    assert info["ns_alg_flops"] == q["ns_alg_flops"]


@pytest.mark.slow
def test_d26_full_stack_sampled():
    # the full d26 stack in the configuration the benchmark times; the oracle
    # checks the first and last layers' six matrices
    p, g, m, _ = workloads.make_stack("d26", "cuda")
    n = len(p)
    run_and_check(p, g, m, check_idx=[0, 4, 5, n - 6, n - 2, n - 1])


def test_many_classes_and_matrices_span_several_launches():
    # 10 distinct oriented shapes (two launch groups of at most 8 classes per GEMM mode) and
    # 200 matrices (two momentum launches of at most 192 matrices)
    base = [(64, 64), (64, 128), (128, 64), (96, 96), (64, 192), (192, 64), (128, 128), (32, 96), (96, 32),
            (160, 160)]
    shapes = [base[i % len(base)] for i in range(200)]
    q = mu.muon_plan_query(shapes, 5)
    assert q["n_classes"] == 10 and q["launches"] == 2 + 3 * 5 * 2
    p, g, m, _ = workloads.make_custom(shapes, "cuda", tag="many")
    run_and_check(p, g, m, check_idx=[0, 1, 5, 9, 10, 99, 150, 191, 192, 199], tol_o=small_side_tol)
    info = mu.muon_get_step_info()
    assert info["launches"] == q["launches"]


@pytest.mark.slow
def test_d26_twenty_carried_steps():
    # the benchmark's run: 20 consecutive d26 steps, momentum carried, a new
    # gradient draw every step.  Every step checks every matrix's momentum
    # against beta m + g (formed in float64 on the device, rounded once); the
    # last step checks all six matrices of layers 0, 13 and 25 (q, k, v, o, the
    # 4:1 MLP input and the 1:4 MLP output) against the oracle run on the state
    # the GPU reached after 19 carried steps
    name = "d26"
    beta = 0.95
    p, g, m, shapes = workloads.make_stack(name, "cuda")
    n = len(p)
    sampled = [6 * layer + k for layer in (0, 13, 25) for k in range(6)]
    assert shapes[sampled[4]] == (6656, 1664) and shapes[sampled[5]] == (1664, 6656)
    steps = 20
    for step in range(steps):
        if step > 0:
            g = [workloads.make_grad(name, i, s, "cuda", 0, step) for i, s in enumerate(shapes)]
        last = step == steps - 1
        if last:
            p0, g0, m0 = (cpu_copy([ts[i] for i in sampled]) for ts in (p, g, m))
        m_prev = [t.clone() for t in m]
        mu.muon_step(p, g, m, lr=0.02, beta=beta, nesterov=True, ns_steps=5)
        mu.muon_get_status()
        bf = float(np.float32(beta))
        for i in range(n):
            exact = (bf * m_prev[i].double() + g[i].double())
            err = (m[i].double() - exact).abs()
            bound = 2.5e-7 * exact.abs() + 1.2e-7 * (bf * m_prev[i].double().abs() + g[i].double().abs())
            assert bool((err <= bound).all()), (step, i)
        del m_prev
        if last:
            for j, i in enumerate(sampled):
                check_matrix(i, p0[j], g0[j], m0[j], p[i].cpu().numpy(), m[i].cpu().numpy(), None,
                             0.02, beta, True, 5, DEFAULT)


def test_sixteen_row_table_runs_sixteen_iterations():
    # the longest table the context takes: 16 rows alternating the default quintic with the
    # cubic Newton-Schulz step (a convergent mix), so every one of the 48 GEMM launches must pick
    # up its own row and the ping-pong buffers alternate through an even count
    cubic = (1.5, -0.5, 0.0)
    rows = [oracle.DEFAULT_ROW if k % 2 == 0 else cubic for k in range(16)]
    mu.muon_destroy()
    mu.muon_init(coeffs=rows, wait_timeout_s=2.0)
    p, g, m, shapes = workloads.make_stack("d2", "cuda")
    assert mu.muon_plan_query(shapes, 16)["launches"] == 1 + 3 * 16
    run_and_check(p, g, m, coeffs=np.array(rows), ns_steps=16)
    assert mu.muon_get_step_info()["launches"] == 1 + 3 * 16


@pytest.mark.parametrize("case", ["d2", "ragged"])
def test_debug_copy_of_o_matches_the_oracle_and_leaves_the_step_unchanged(case):
    # MUON_DEBUG_KEEP_O adds an fp32 store of O to the last launch (and runs its ring with one stage
    # fewer to make room).  The copy must match the oracle, and the weights and momentum must come
    # out bit for bit as in the plain step on the same inputs.
    if case == "d2":
        p, g, m, _ = workloads.make_stack("d2", "cuda")
        tol = None
    else:
        p, g, m, _ = workloads.make_custom(RAGGED, "cuda", tag="ragged")
        tol = small_side_tol
    snap = [t.clone() for t in p + g + m]
    run_gpu_step(p, g, m)
    plain = [t.clone() for t in p + m]
    mu.muon_destroy()
    mu.muon_init(debug_flags=mu.MUON_DEBUG_KEEP_O, wait_timeout_s=2.0)
    for dst, src in zip(p + g + m, snap):
        dst.copy_(src)
    run_and_check(p, g, m, keep_o=True, tol_o=tol)
    for a, b in zip(plain, p + m):
        assert torch.equal(a, b)


def test_several_shape_lists_keep_their_workspaces():
    # the context keeps a workspace per shape list (up to 8): alternating lists must give the
    # oracle's result every time, and a ninth list (dropping the least recently used) too
    lists = [[(64, 64), (128, 64)], [(64, 128)], [(96, 96), (64, 64)], [(128, 128)], [(64, 192)], [(192, 64)],
             [(160, 160)], [(72, 72)], [(64, 64), (64, 64), (128, 128)]]
    # lists 0..7 fill the cache; list 8 then drops the least recently used, list 2; 0 is still held,
    # 2 is rebuilt
    order = [0, 1, 2, 0, 1, 3, 4, 5, 6, 7, 8, 0, 2]
    for step, k in enumerate(order):
        p, g, m, _ = workloads.make_custom(lists[k], "cuda", tag=f"plans{step}")
        run_and_check(p, g, m, ns_steps=3)
