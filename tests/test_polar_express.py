"""Pins of the derived Polar Express coefficient table (oracle/polar_express.py), CPU only.

The pages print two of the five rows (to three decimals) and elide the rest;
the table is derived by the Polar Express construction with the readings stated
in oracle/polar_express.py.  What pins it to something other than itself:

* the two printed rows ("Cara Melatih ChatGPT Sendiri dengan Budget 50 Dolar",
  section "2. Pengoptimal Muon (nanochat/optim.py)", coefficient list);
* the Chebyshev alternation theorem: an odd quintic (three free coefficients)
  is the best max-norm approximation of 1 on an interval exactly when its
  error reaches its maximum with alternating signs at four points, so each
  fitted polynomial is checked for that, on a dense grid;
* an independent solver: the same minimax problem as a linear program on a
  grid (scipy's HiGHS), which must give the same error;
* the limit of a shrinking interval (p(1) = 1, p'(1) = p''(1) = 0);
* the construction's own guarantee: after t rows every x in [l_0, 1] lies in
  the t-th interval, and the last row's band is centred on 1;
* the oracle's loop with the table follows the closed form U f(S) V^T.

``test_pins_catch_planted_mistakes`` re-runs the pins on mutated copies of the
construction and checks that each fails at least one.
"""
import os
import types

import numpy as np
import pytest

import oracle
import oracle.polar_express as pe

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "polar_express_rows.txt")
PRINTED = oracle.PAGES_POLAR_EXPRESS_ROWS   # (8.156, -22.483, 15.879), (4.043, -2.809, 0.500)


def _golden_rows():
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    return np.array([[float(v) for v in r[:3]] for r in rows]), np.array([[float(v) for v in r[3:]] for r in rows])


# ---------------------------------------------------------------- checks (run on a construction module)
def check_printed_rows(mod):
    rows, _ = mod.polar_express_rows()
    diff = np.abs(np.array(rows[:2]) - PRINTED)
    # every printed figure within one unit of its last decimal ...
    assert np.all(diff < 1e-3), diff
    # ... and all but the first row's leading term (8.15655 printed as 8.156) round to it
    mask = np.ones_like(diff, dtype=bool)
    mask[0, 0] = False
    assert np.all(diff[mask] <= 5e-4), diff


def check_equioscillation(mod):
    rows, intervals = mod.polar_express_rows()
    for t, (lo, hi) in enumerate(intervals):
        flo = max(lo, mod.CUSHION * hi)
        a, b, c, E = mod.minimax_odd_quintic(flo, hi)
        xs = np.linspace(flo, hi, 400001)
        err = 1.0 - mod.quintic(xs, (a, b, c))
        assert abs(np.abs(err).max() - E) <= 1e-10 * max(E, 1.0), t
        # alternation: +E at flo, -E, +E at the interior extrema, -E at hi
        d = np.sign(np.diff(err))
        turns = xs[1:-1][d[1:] != d[:-1]]
        assert len(turns) == 2, (t, turns)
        pts = [flo, *turns, hi]
        vals = 1.0 - mod.quintic(np.array(pts), (a, b, c))
        assert np.allclose(vals, [E, -E, E, -E], rtol=0, atol=1e-7), (t, vals, E)
        # the table row is that polynomial, recentred on the true interval (and, except for the
        # last row, with x replaced by x / safety): same shape (c/a)/(b/a)^2 up to the safety
        ra, rb, rc = rows[t]
        sf = mod.SAFETY if t < len(rows) - 1 else 1.0
        assert np.isclose((rc / ra) / (rb / ra) ** 2, (c / a) / (b / a) ** 2, rtol=1e-12), t
        assert np.isclose((rb / ra) * sf ** 2, b / a, rtol=1e-12), t


def check_intervals_and_band(mod):
    rows, intervals = mod.polar_express_rows()
    xs = np.geomspace(mod.L0, 1.0, 200001)
    f = xs.copy()
    for t, row in enumerate(rows):
        lo, hi = intervals[t]
        assert f.min() >= lo * (1 - 1e-12) and f.max() <= hi * (1 + 1e-12), t
        f = mod.quintic(f, row)
    # the last row's band is centred on 1 ([l, 2 - l] with l the image of the lower end)
    assert np.isclose(f.min() + f.max(), 2.0, rtol=0, atol=1e-9), (f.min(), f.max())
    assert 0.85 < f.min() < 0.87


def check_limit_polynomial(mod):
    a, b, c, E = mod.minimax_odd_quintic(1.0 - 1e-9, 1.0)
    assert E == 0.0
    assert np.isclose(a + b + c, 1.0) and np.isclose(a + 3 * b + 5 * c, 0.0) and np.isclose(6 * b + 20 * c, 0.0)


CHECKS = [check_printed_rows, check_equioscillation, check_intervals_and_band, check_limit_polynomial]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check(pe)


@pytest.mark.parametrize("lo,hi", [(0.02, 1.0), (0.3, 1.0), (0.0408, 1.9918), (0.4, 1.6)])
def test_remez_agrees_with_a_linear_program(lo, hi):
    # min E subject to |1 - (a x + b x^3 + c x^5)| <= E on a fine grid: a different algorithm for
    # the same minimax problem
    from scipy.optimize import linprog
    xs = np.linspace(lo, hi, 4001)
    V = np.stack([xs, xs ** 3, xs ** 5], axis=1)
    ones = np.ones((len(xs), 1))
    A_ub = np.vstack([np.hstack([-V, -ones]), np.hstack([V, -ones])])
    b_ub = np.concatenate([-np.ones(len(xs)), np.ones(len(xs))])
    res = linprog(c=[0, 0, 0, 1], A_ub=A_ub, b_ub=b_ub, bounds=[(None, None)] * 4, method="highs")
    assert res.status == 0
    a, b, c, E = pe.minimax_odd_quintic(lo, hi)
    assert abs(res.x[3] - E) <= 1e-6 * E + 1e-9, (res.x[3], E)
    assert np.allclose(res.x[:3], [a, b, c], rtol=1e-4, atol=1e-6), (res.x[:3], (a, b, c))


def test_golden_table_is_the_construction():
    rows, intervals = pe.polar_express_rows()
    g_rows, g_iv = _golden_rows()
    assert g_rows.shape == (5, 3)
    assert np.array_equal(g_rows, np.array(rows)) and np.array_equal(g_iv, np.array(intervals))


def test_binding_table_is_the_golden_table():
    import pretraining_optimizer_step_b300 as mu
    g_rows, _ = _golden_rows()
    assert np.array_equal(np.array(mu.POLAR_EXPRESS_COEFFS, dtype=np.float64), g_rows)


def test_oracle_loop_with_the_table_follows_the_closed_form_and_band():
    rows, _ = pe.polar_express_rows()
    rng = np.random.default_rng(21)
    for shape in [(8, 8), (12, 30), (30, 12), (48, 48)]:
        # singular values spread over [1e-3, 1] relative to the largest
        U, _ = np.linalg.qr(rng.standard_normal((shape[0], shape[0])))
        V, _ = np.linalg.qr(rng.standard_normal((shape[1], shape[1])))
        k = min(shape)
        s = np.geomspace(1.0, 1e-3, k)
        G = (U[:, :k] * s) @ V[:, :k].T
        O = oracle.orthogonalize(G, np.array(rows), eps=0.0)
        fro = np.linalg.norm(G)
        x = s / fro
        for row in rows:
            x = pe.quintic(x, row)
        ref = (U[:, :k] * x) @ V[:, :k].T
        assert np.linalg.norm(O - ref) <= 1e-10 * np.linalg.norm(ref), shape
        # no output singular value leaves the table's band from above (below 1e-3 the
        # composition stays under its value at 1e-3)
        so = np.linalg.svd(O, compute_uv=False)
        assert so.max() <= 1.1412, shape


# ---------------------------------------------------------------- planted mistakes
MUTANTS = {
    "no_cushion": ("minimax_odd_quintic(max(lo, cushion * hi), hi)", "minimax_odd_quintic(lo, hi)"),
    "no_recentring": ("k = 2.0 / (quintic(lo, (a, b, c)) + quintic(hi, (a, b, c)))", "k = 1.0"),
    "safety_on_every_row": ("sf = safety if len(rows) < n_rows - 1 else 1.0", "sf = safety"),
    "no_safety": ("sf = safety if len(rows) < n_rows - 1 else 1.0", "sf = 1.0"),
    "safety_as_multiplier": ("row = (a * k / sf, b * k / sf ** 3, c * k / sf ** 5)",
                             "row = (a * k * sf, b * k * sf ** 3, c * k * sf ** 5)"),
    "upper_end_is_its_image": ("        hi = 2.0 - lo\n", "        hi = float(quintic(hi, row))\n"),
    "lower_end_not_updated": ("        lo = float(quintic(lo, row))\n        hi = 2.0 - lo\n",
                              "        hi = 2.0 - float(quintic(lo, row))\n"),
    "alternation_sign_flipped": ("(-1.0) ** i] for i, x in enumerate(pts)", "(-1.0) ** (i // 2)] for i, x in enumerate(pts)"),
    "wrong_critical_points": ("(10.0 * c)", "(5.0 * c)"),
}


def _mutant_module(old, new):
    src = open(pe.__file__).read()
    assert src.count(old) >= 1, old
    mod = types.ModuleType("pe_mutant")
    exec(compile(src.replace(old, new), "pe_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name):
    old, new = MUTANTS[name]
    failed = []
    with np.errstate(all="ignore"):
        try:
            mod = _mutant_module(old, new)
        except Exception as exc:  # a mutant may not even import
            failed.append(("import", str(exc)[:60]))
            mod = None
        if mod is not None:
            for check in CHECKS:
                try:
                    check(mod)
                except (AssertionError, ArithmeticError, ValueError, np.linalg.LinAlgError, FloatingPointError) as exc:
                    failed.append((check.__name__, str(exc)[:60]))
    assert failed, f"mutant {name} passed every pin"
