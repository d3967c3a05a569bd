"""Pins of the fp64 oracle to facts outside itself (CPU only).

The oracle restates the Muon step of "Cara Melatih ChatGPT Sendiri dengan Budget
50 Dolar" (apidog.com), section "2. Pengoptimal Muon (nanochat/optim.py)".  The
pages print no input/output example for it, so the pins come from mathematics:

* closed form: for G = U S V^T, K iterations give U f(S/(||G||_F+eps)) V^T with
  f the K-fold composition of x -> a x + b x^3 + c x^5 (LAPACK SVD via numpy);
* the output band of the default table on well-conditioned inputs;
* exactly orthogonal inputs stay on their direction, scaled by f(1/sqrt(n));
* hand-worked single iterations (tests/golden/hand_iteration.txt);
* 1 x n inputs reduce to the scalar map; orientation and scale symmetries;
* momentum special cases and the aspect-ratio update scale.

``test_pins_catch_planted_mistakes`` compiles mutated copies of the oracle source
(dropped term, wrong sign, swapped coefficient, transposed operand, ...) and
checks that each one fails at least one pin.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FIXED = oracle.DEFAULT_ROW


def scalar_map(x, rows):
    """f = phi_K o ... o phi_1 evaluated on numbers (the closed form's scalar part)."""
    x = np.asarray(x, dtype=np.float64)
    for a, b, c in rows:
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def closed_form(G, rows, eps):
    U, S, Vt = np.linalg.svd(G, full_matrices=False)
    fro = np.sqrt(np.sum(G.astype(np.float64) ** 2))
    return (U * scalar_map(S / (fro + eps), rows)) @ Vt


def default_band():
    xs = np.linspace(0.01, 1.0, 200001)
    f = scalar_map(xs, [FIXED] * 5)
    return f.min(), f.max()


SHAPES = [(2, 2), (3, 5), (5, 3), (8, 8), (16, 64), (64, 16), (24, 40), (1, 7), (7, 1)]
MIXED_ROWS = [tuple(r) for r in oracle.PAGES_POLAR_EXPRESS_ROWS] + [FIXED] * 3


# ---------------------------------------------------------------- pin checks
# Each check raises AssertionError on failure; the tests below run them on the
# real oracle, and the mutation test runs them on planted mistakes.

def check_closed_form():
    rng = np.random.default_rng(1)
    for rows in ([FIXED] * 5, MIXED_ROWS, [FIXED]):
        for shape in SHAPES:
            G = rng.standard_normal(shape)
            O = oracle.orthogonalize(G, rows, eps=1e-7)
            ref = closed_form(G, rows, 1e-7)
            err = np.linalg.norm(O - ref) / max(np.linalg.norm(ref), 1e-300)
            assert err < 1e-10, (shape, err)


def check_closed_form_nonnormal_square():
    # a non-normal square input separates X p(X^T X) from p(X X^T)-style mistakes
    G = np.triu(np.arange(1.0, 37.0).reshape(6, 6)) + 0.1 * np.eye(6)
    O = oracle.orthogonalize(G, [FIXED] * 3, eps=0.0)
    ref = closed_form(G, [FIXED] * 3, 0.0)
    assert np.linalg.norm(O - ref) / np.linalg.norm(ref) < 1e-10


def check_band():
    lo, hi = default_band()
    rng = np.random.default_rng(2)
    for shape in [(8, 8), (6, 20), (20, 6), (16, 48)]:
        for _ in range(5):
            G = rng.standard_normal(shape)
            s = np.linalg.svd(G, compute_uv=False)
            if s.min() / np.linalg.norm(G) < 0.01:
                continue
            O = oracle.orthogonalize(G, oracle.DEFAULT_COEFFS)
            so = np.linalg.svd(O, compute_uv=False)
            assert so.min() >= lo - 1e-9 and so.max() <= hi + 1e-9, (shape, so.min(), so.max())
            U, _, Vt = np.linalg.svd(G, full_matrices=False)
            assert np.linalg.norm(O - U @ Vt, 2) <= 0.32


def check_orthogonal_input():
    rng = np.random.default_rng(3)
    for n in (2, 5, 16, 40):
        Q, _ = np.linalg.qr(rng.standard_normal((n, n)))
        O = oracle.orthogonalize(Q, oracle.DEFAULT_COEFFS, eps=0.0)
        expect = scalar_map(1.0 / np.sqrt(n), [FIXED] * 5)
        assert np.abs(O - expect * Q).max() < 1e-12, n


def check_hand_iteration():
    path = os.path.join(GOLDEN, "hand_iteration.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert rows
    for name, a, b, c, y3, y4 in rows:
        G = np.diag([3.0, 4.0])
        O = oracle.orthogonalize(G, [(float(a), float(b), float(c))], eps=0.0)
        assert abs(O[0, 0] - float(y3)) < 1e-12 and abs(O[1, 1] - float(y4)) < 1e-12, name
        assert abs(O[0, 1]) < 1e-15 and abs(O[1, 0]) < 1e-15


def check_row_vector():
    rng = np.random.default_rng(4)
    for n in (1, 7, 64):
        g = rng.standard_normal((1, n))
        nrm = np.linalg.norm(g)
        O = oracle.orthogonalize(g, oracle.DEFAULT_COEFFS, eps=1e-7)
        expect = scalar_map(nrm / (nrm + 1e-7), [FIXED] * 5) * g / nrm
        assert np.abs(O - expect).max() < 1e-12
        Ot = oracle.orthogonalize(g.T, oracle.DEFAULT_COEFFS, eps=1e-7)
        assert np.abs(Ot - expect.T).max() < 1e-12


def check_orientation_and_scale():
    rng = np.random.default_rng(5)
    G = rng.standard_normal((12, 30))
    O = oracle.orthogonalize(G)
    Ot = oracle.orthogonalize(np.ascontiguousarray(G.T))
    assert np.array_equal(Ot, O.T)
    O5 = oracle.orthogonalize(G * 1e-3, eps=0.0)
    O6 = oracle.orthogonalize(G * 7.5, eps=0.0)
    assert np.abs(O5 - O6).max() < 1e-12


def check_momentum():
    rng = np.random.default_rng(6)
    g = rng.standard_normal((4, 8)).astype(np.float32)
    m = rng.standard_normal((4, 8)).astype(np.float32)
    g64, m64 = g.astype(np.float64), m.astype(np.float64)
    # beta = 0: the direction is the gradient
    mo, u = oracle.momentum(g, m, 0.0, True)
    assert np.array_equal(mo, g) and np.array_equal(u, g64)
    # g = 0 with Nesterov: m' = beta m, u = beta^2 m
    z = np.zeros_like(g)
    mo, u = oracle.momentum(z, m, 0.5, True)
    assert np.array_equal(mo, (0.5 * m64).astype(np.float32))
    assert np.allclose(u, 0.25 * m64, rtol=0, atol=1e-15)
    # plain heavy ball: u = m' = beta m + g
    mo, u = oracle.momentum(g, m, 0.9, False)
    assert np.allclose(u, 0.9 * m64 + g64, rtol=0, atol=1e-12)
    assert np.array_equal(mo, u.astype(np.float32))
    # Nesterov: u = g + beta m'
    mo, u = oracle.momentum(g, m, 0.9, True)
    assert np.allclose(u, g64 + 0.9 * (0.9 * m64 + g64), rtol=0, atol=1e-12)


def _constant_gradient_run(g, beta, mode, nesterov, steps):
    """Momentum states m_1..m_k and directions u_0..u_{k-1} from m_0 = 0 under a constant g."""
    m = np.zeros_like(g)
    ms, us = [], []
    for _ in range(steps):
        m, u = oracle.momentum(g, m, beta, nesterov, mode=mode)
        ms.append(m.astype(np.float64))
        us.append(u)
    return ms, us


def check_momentum_transients():
    # Facts about both momentum forms that do not restate their update rule:
    #  * from m = 0 under a constant gradient g, the heavy-ball buffer is the partial geometric
    #    sum m_k = g (1 - beta^k) / (1 - beta), and the EMA buffer is its (1 - beta)-weighted
    #    form m_k = g (1 - beta^k) (the bias the usual EMA correction divides out);
    #  * Nesterov looks one step ahead: under a constant gradient the direction of step k is the
    #    buffer the next step will hold, u_k = m_{k+1} (plain momentum: u_k = m_k);
    #  * the EMA buffer started at m = g stays at g, and beta = 0 gives m' = u = g.
    rng = np.random.default_rng(8)
    g = rng.standard_normal((3, 8)).astype(np.float32)
    g64 = g.astype(np.float64)
    beta = 0.9
    steps = 6
    for mode in (0, 1):
        for nesterov in (False, True):
            ms, us = _constant_gradient_run(g, beta, mode, nesterov, steps + 1)
            for k in range(1, steps + 1):
                geo = (1.0 - beta ** k) / (1.0 - beta)
                expect = g64 * (geo if mode == 0 else (1.0 - beta ** k))
                assert np.allclose(ms[k - 1], expect, rtol=1e-6, atol=1e-7), (mode, nesterov, k)
            for k in range(steps):
                ahead = ms[k + 1] if nesterov else ms[k]
                assert np.allclose(us[k], ahead, rtol=1e-6, atol=1e-7), (mode, nesterov, k)
    for nesterov in (False, True):
        mo, u = oracle.momentum(g, g.copy(), 0.75, nesterov, mode=1)
        assert np.allclose(mo, g64, rtol=1e-7, atol=0) and np.allclose(u, g64, rtol=1e-7, atol=0)
        mo, u = oracle.momentum(g, rng.standard_normal(g.shape).astype(np.float32), 0.0, nesterov, mode=1)
        assert np.array_equal(mo, g) and np.allclose(u, g64, rtol=0, atol=0)


def check_update_scale():
    rng = np.random.default_rng(7)
    for (r, c), s in (((512, 128), 2.0), ((128, 512), 1.0), ((64, 64), 1.0), ((72, 8), 3.0)):
        p = rng.standard_normal((r, c)).astype(np.float32)
        g = rng.standard_normal((r, c)).astype(np.float32)
        m = rng.standard_normal((r, c)).astype(np.float32)
        p1, m1, O = oracle.muon_matrix(p, g, m, lr=0.02, beta=0.95, nesterov=True, ns_steps=2)
        expect = (p.astype(np.float64) - 0.02 * s * O).astype(np.float32)
        assert np.array_equal(p1, expect), (r, c)
        _, u = oracle.momentum(g, m, 0.95, True)
        assert np.abs(O - oracle.orthogonalize(u, ns_steps=2)).max() == 0.0


PIN_CHECKS = [check_closed_form, check_closed_form_nonnormal_square, check_band,
              check_orthogonal_input, check_hand_iteration, check_row_vector,
              check_orientation_and_scale, check_momentum, check_momentum_transients, check_update_scale]


@pytest.mark.parametrize("check", PIN_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def test_default_band_matches_quoted_band():
    # the method's description quotes an output band of about [0.68, 1.13]
    lo, hi = default_band()
    assert 0.675 < lo < 0.69 and 1.125 < hi < 1.14


def test_orthogonal_scale_values():
    # f(1/sqrt(n)) for the default table at the orthogonal-input sizes used above
    # and at d26's width; evaluated on numbers, independent of the matrix code
    got = [float(scalar_map(1 / np.sqrt(n), [FIXED] * 5)) for n in (2, 128, 768, 1664)]
    assert np.allclose(got, [1.1081111, 0.7227622, 1.0835946, 0.9015170], atol=1e-7)


# ---------------------------------------------------------------- planted mistakes
MUTANTS = {
    "drop_c_term": ("b * A[e] + c * AA[e]", "b * A[e]"),
    "axpy_sign": ("a * X[e] + BX[e]", "a * X[e] - BX[e]"),
    "b_c_swapped": ("c = coeffs[3 * k + 2]", "c = coeffs[3 * k + 1]"),
    "a_from_b": ("const double a = coeffs[3 * k]", "const double a = coeffs[3 * k + 1]"),
    "right_multiply": ("mat_mul(rows, cols, rows, A, X, BX)", "mat_mul(rows, cols, cols, X, A, BX)"),
    "gram_transposed": ("mat_mul(rows, rows, cols, X, XT, A)", "mat_mul(rows, rows, cols, XT, X, A)"),
    "no_normalise": ("for (size_t e = 0; e < rc; ++e) X[e] *= s;", ""),
    "no_eps": ("oracle_frobenius((long)rc, X) + eps)", "oracle_frobenius((long)rc, X))"),
    "no_transpose_back": ("if (tall) transpose(rows, cols, X, O);", "if (0) {}"),
    "aspect_inverted": ("(double)r / (double)c", "(double)c / (double)r"),
    "nesterov_uses_old_m": ("u = nesterov ? gd + beta * mn : mn", "u = nesterov ? gd + beta * md : mn"),
    "momentum_no_beta": ("mn = beta * md + gd", "mn = md + gd"),
    "ema_no_one_minus_beta": ("mn = beta * md + (1.0 - beta) * gd", "mn = beta * md + gd"),
    "ema_weights_swapped": ("mn = beta * md + (1.0 - beta) * gd", "mn = (1.0 - beta) * md + beta * gd"),
    "ema_nesterov_uses_old_m": ("u = nesterov ? (1.0 - beta) * gd + beta * mn : mn",
                                "u = nesterov ? (1.0 - beta) * gd + beta * md : mn"),
    "loop_one_short": ("for (int k = 0; k < K; ++k)", "for (int k = 1; k < K; ++k)"),
}


def _run_pins():
    failed = []
    for check in PIN_CHECKS:
        try:
            check()
        except (AssertionError, ValueError, np.linalg.LinAlgError) as exc:
            failed.append((check.__name__, str(exc)[:80]))
    return failed


def _scratch_dir():
    """Build folder for throwaway mutant libraries, inside the repository (git-ignored)."""
    d = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "_build", "tests")
    os.makedirs(d, exist_ok=True)
    return d

@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = MUTANTS[name]
    src = open(oracle.source_path()).read()
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    with tempfile.TemporaryDirectory(dir=_scratch_dir()) as tmp:
        c_path = os.path.join(tmp, "mutant.c")
        so_path = os.path.join(tmp, "libmutant.so")
        open(c_path, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", so_path,
                        c_path, "-lm"], check=True)
        # a mutant may overflow (no normalisation, say): numpy's warnings are expected there
        with oracle.using_library(so_path), np.errstate(all="ignore"):
            failed = _run_pins()
    assert failed, f"mutant {name} passed every pin"


@pytest.mark.parametrize("shape", [(48, 48), (64, 200), (200, 64), (8, 96)])
def test_closed_form_helper_matches_the_oracle(shape):
    # the closed form the large GPU cases are checked against agrees with the
    # step-by-step oracle (both fp64) on shapes the oracle finishes at once
    from closed_form import closed_form_o
    rng = np.random.default_rng(sum(shape))
    g = (rng.standard_normal(shape) * 1e-3).astype(np.float32)
    m = (rng.standard_normal(shape) * 1e-3).astype(np.float32)
    p = (rng.standard_normal(shape) * 0.05).astype(np.float32)
    _, _, O = oracle.muon_matrix(p, g, m, lr=np.float32(0.02), beta=np.float32(0.95), nesterov=True, ns_steps=5)
    ref = closed_form_o(g, m, 0.95, oracle.DEFAULT_COEFFS)
    assert np.linalg.norm(ref - O) <= 1e-10 * np.linalg.norm(O)
