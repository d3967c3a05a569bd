"""Pins of the AdamW oracle (CPU only).

The optimizer split on the dev.to page (section "2. ตัวปรับปรุง Muon", optimizer
table) sends embeddings, lm_head and scalar parameters to AdamW; the pages give
no formula, so the oracle takes decoupled weight decay with bias-corrected
moments.  The pins: hand-worked steps (tests/golden/adamw_hand.txt), the
first-step sign law, the weight-decay-only and zero-learning-rate cases, the
steady state of the moments under a constant gradient, and planted mistakes.
"""
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "adamw_hand.txt")


def check_hand_rows():
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for name, p, g, m, v, lr, b1, b2, eps, wd, t, p_out, m_out, v_out in rows:
        P, M, V = oracle.adamw(np.float32([p]), np.float32([g]), np.float32([m]), np.float32([v]), float(lr),
                               float(b1), float(b2), float(eps), float(wd), int(t))
        # stored as float32: compare within one float32 rounding of the exact value
        for got, want in ((P[0], p_out), (M[0], m_out), (V[0], v_out)):
            want = float(want)
            assert abs(float(got) - want) <= 1e-6 * max(1.0, abs(want)), (name, got, want)


def check_first_step_is_signed_lr():
    rng = np.random.default_rng(11)
    g = rng.standard_normal(1000).astype(np.float32)
    g[g == 0] = 1.0
    p = rng.standard_normal(1000).astype(np.float32)
    z = np.zeros_like(p)
    P, M, V = oracle.adamw(p, g, z, z, lr=0.003, beta1=0.8, beta2=0.95, eps=0.0, weight_decay=0.0, step=1)
    assert np.allclose(P, p - 0.003 * np.sign(g), rtol=0, atol=2e-7)
    assert np.allclose(M, 0.2 * g.astype(np.float64), rtol=1e-6)
    assert np.allclose(V, 0.05 * g.astype(np.float64) ** 2, rtol=1e-6)


def check_zero_lr_and_decay_only():
    rng = np.random.default_rng(12)
    p = rng.standard_normal(64).astype(np.float32)
    g = rng.standard_normal(64).astype(np.float32)
    m = rng.standard_normal(64).astype(np.float32) * 0.1
    v = np.abs(rng.standard_normal(64)).astype(np.float32)
    P, _, _ = oracle.adamw(p, g, m, v, lr=0.0, weight_decay=0.3, step=5)
    assert np.array_equal(P, p)
    # a zero gradient with zero moments: only the decay acts (the m term is exactly 0)
    z = np.zeros_like(p)
    P, M, V = oracle.adamw(p, z, z, z, lr=0.1, weight_decay=0.5, eps=1e-8, step=3)
    assert np.allclose(P, p.astype(np.float64) * 0.95, rtol=1e-7, atol=0)
    assert not M.any() and not V.any()


def check_constant_gradient_steady_state():
    # with the same gradient every step the bias-corrected moments equal g and g^2 at
    # every t, so every step moves p by lr * sign(g) (eps = 0, wd = 0)
    p = np.float32([0.5, -2.0, 3.0])
    g = np.float32([0.25, -4.0, 1e-3])
    m = np.zeros(3, np.float32)
    v = np.zeros(3, np.float32)
    for t in range(1, 6):
        p, m, v = oracle.adamw(p, g, m, v, lr=0.01, beta1=0.9, beta2=0.99, eps=0.0, step=t)
    assert np.allclose(p, np.float32([0.5, -2.0, 3.0]) - 5 * 0.01 * np.sign(g), rtol=0, atol=2e-6)


def check_eps_bounds_the_step():
    # g = 0, v = 0, m = 0.5 at t = 1 (beta1 0.9, beta2 0.999, lr 0.1, eps 0.01):
    # m' = 0.45, v' = 0, m_hat = 0.45 / 0.1 = 4.5, v_hat = 0, so the step is 4.5 / (0 + 0.01) = 450 * 0.1 = 45
    P, M, V = oracle.adamw(np.float32([0.0]), np.float32([0.0]), np.float32([0.5]), np.float32([0.0]),
                           lr=0.1, beta1=0.9, beta2=0.999, eps=0.01, weight_decay=0.0, step=1)
    assert abs(float(P[0]) + 45.0) < 1e-4 and abs(float(M[0]) - 0.45) < 1e-7 and V[0] == 0.0


PIN_CHECKS = [check_hand_rows, check_eps_bounds_the_step, check_first_step_is_signed_lr, check_zero_lr_and_decay_only,
              check_constant_gradient_steady_state]


@pytest.mark.parametrize("check", PIN_CHECKS, ids=lambda f: f.__name__)
def test_adamw_pin(check):
    check()


MUTANTS = {
    "no_bias_correction1": ("pd -= (lr / bc1) * md", "pd -= lr * md"),
    "no_bias_correction2": ("sqrt(vd / bc2)", "sqrt(vd)"),
    "eps_inside_sqrt": ("sqrt(vd / bc2) + eps", "sqrt(vd / bc2 + eps)"),
    "coupled_decay": ("(double)p[e] * (1.0 - lr * weight_decay)", "(double)p[e] * (1.0 - weight_decay)"),
    "m_weights_swapped": ("beta1 * (double)m[e] + (1.0 - beta1) * gd", "(1.0 - beta1) * (double)m[e] + beta1 * gd"),
    "v_not_squared": ("(1.0 - beta2) * gd * gd", "(1.0 - beta2) * fabs(gd)"),
    "step_sign": ("pd -= (lr / bc1)", "pd += (lr / bc1)"),
}


def _scratch_dir():
    """Build folder for throwaway mutant libraries, inside the repository (git-ignored)."""
    d = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "_build", "tests")
    os.makedirs(d, exist_ok=True)
    return d

@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_adamw_pins_catch_planted_mistakes(name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = MUTANTS[name]
    src = open(oracle.source_path()).read()
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    with tempfile.TemporaryDirectory(dir=_scratch_dir()) as tmp:
        c_path = os.path.join(tmp, "mutant.c")
        so_path = os.path.join(tmp, "libmutant.so")
        open(c_path, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", so_path, c_path, "-lm"],
                       check=True)
        failed = []
        with oracle.using_library(so_path):
            for check in PIN_CHECKS:
                try:
                    check()
                except AssertionError as exc:
                    failed.append(check.__name__)
    assert failed, f"mutant {name} passed every AdamW pin"
