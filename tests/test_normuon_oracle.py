"""Pins of the NorMuon oracle (CPU only).

The pages sketch NorMuon as a per-neuron rescale after orthogonalisation
(apidog.com section "2. Pengoptimal Muon", paragraph "Reduksi Varians NorMuon";
dev.to "NorMuon variance scaling") and leave red_dim, the second-moment state,
step_size and v_norm_new undefined.  The reading pinned here: a neuron is a
stored row, V <- beta2 V + (1 - beta2) mean_j O_ij^2, step = 1 / sqrt(V + eps),
and the rows are rescaled by step * v_norm / v_norm_new, which keeps ||O||_F.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "normuon_hand.txt")


def check_hand_example():
    vals = [float(x) for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#") for x in ln.split()]
    O, V = oracle.normuon_scale(np.array([[3.0, 4.0], [1.0, 0.0]]), np.zeros(2), beta2=0.0, eps=0.0)
    assert np.allclose(O.reshape(-1), vals[:4], rtol=0, atol=1e-9)
    assert np.allclose(V, vals[4:], rtol=0, atol=0)


def check_norm_is_preserved():
    rng = np.random.default_rng(21)
    for shape in [(5, 9), (9, 5), (16, 16), (1, 7)]:
        O = rng.standard_normal(shape) * rng.uniform(0.1, 3.0, size=(shape[0], 1))
        V = np.abs(rng.standard_normal(shape[0])).astype(np.float32) * 0.1
        O2, _ = oracle.normuon_scale(O, V, beta2=0.9, eps=1e-8)
        assert abs(np.linalg.norm(O2) - np.linalg.norm(O)) < 1e-12 * np.linalg.norm(O), shape


def check_equal_rows_are_left_alone():
    # rows of equal mean square and a uniform state: every row gets the same scale, which the
    # norm constraint fixes at 1
    rng = np.random.default_rng(22)
    Q, _ = np.linalg.qr(rng.standard_normal((12, 12)))
    V = np.full(12, 0.3, np.float32)
    O2, V2 = oracle.normuon_scale(Q, V, beta2=0.5, eps=1e-8)
    assert np.abs(O2 - Q).max() < 1e-12
    assert np.allclose(V2, np.float32(0.5 * 0.3 + 0.5 / 12), rtol=1e-6)


def check_fresh_state_equalises_rows():
    # beta2 = 0 and eps = 0: step_i = 1 / sqrt(v_mean_i), so every row ends with the same
    # mean square, ||O||^2 / (r c)
    rng = np.random.default_rng(23)
    O = rng.standard_normal((6, 10)) * np.arange(1, 7)[:, None]
    O2, _ = oracle.normuon_scale(O, np.zeros(6), beta2=0.0, eps=0.0)
    row_ms = (O2 ** 2).mean(axis=1)
    assert np.allclose(row_ms, (O ** 2).sum() / O.size, rtol=1e-12)


def check_state_update():
    rng = np.random.default_rng(24)
    O = rng.standard_normal((4, 6))
    V = np.float32([0.5, 0.0, 2.0, 1e-3])
    _, V2 = oracle.normuon_scale(O, V, beta2=0.8, eps=1e-8)
    want = (0.8 * V.astype(np.float64) + 0.2 * (O ** 2).mean(axis=1)).astype(np.float32)
    assert np.array_equal(V2, want)


def check_single_row_is_unchanged():
    O = np.array([[0.3, -1.2, 2.5]])
    O2, _ = oracle.normuon_scale(O, np.float32([0.7]), beta2=0.9, eps=1e-6)
    assert np.abs(O2 - O).max() < 1e-14


def check_matrix_step_uses_scaled_update():
    rng = np.random.default_rng(25)
    p = rng.standard_normal((24, 8)).astype(np.float32)
    g = rng.standard_normal((24, 8)).astype(np.float32)
    m = rng.standard_normal((24, 8)).astype(np.float32)
    V = np.abs(rng.standard_normal(24)).astype(np.float32)
    p1, m1, V1, O1 = oracle.normuon_matrix(p, g, m, V, lr=0.02, beta=0.95, ns_steps=3)
    _, u = oracle.momentum(g, m, 0.95, True)
    O, V_ref = oracle.normuon_scale(oracle.orthogonalize(u, ns_steps=3), V)
    assert np.abs(O1 - O).max() == 0.0 and np.array_equal(V1, V_ref)
    assert np.array_equal(p1, (p.astype(np.float64) - 0.02 * np.sqrt(3.0) * O).astype(np.float32))


PIN_CHECKS = [check_hand_example, check_norm_is_preserved, check_equal_rows_are_left_alone,
              check_fresh_state_equalises_rows, check_state_update, check_single_row_is_unchanged,
              check_matrix_step_uses_scaled_update]


@pytest.mark.parametrize("check", PIN_CHECKS, ids=lambda f: f.__name__)
def test_normuon_pin(check):
    check()


MUTANTS = {
    "no_norm_ratio": ("*= st[i] * ratio;", "*= st[i];"),
    "v_weights_swapped": ("beta2 * (double)V[i] + (1.0 - beta2) * vm[i]", "(1.0 - beta2) * (double)V[i] + beta2 * vm[i]"),
    "step_without_sqrt": ("st[i] = 1.0 / sqrt(Vn + eps);", "st[i] = 1.0 / (Vn + eps);"),
    "new_norm_without_square": ("s_new += vm[i] * st[i] * st[i];", "s_new += vm[i] * st[i];"),
    "sum_not_mean": ("vm[i] = s / (double)c;", "vm[i] = s;"),
    "old_state_stored": ("V[i] = (float)Vn;", "(void)Vn;"),
}


def _scratch_dir():
    """Build folder for throwaway mutant libraries, inside the repository (git-ignored)."""
    d = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "_build", "tests")
    os.makedirs(d, exist_ok=True)
    return d

@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_normuon_pins_catch_planted_mistakes(name):
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
                except AssertionError:
                    failed.append(check.__name__)
    assert failed, f"mutant {name} passed every NorMuon pin"
