"""Per-iteration "Polar Express" coefficient rows for the Newton-Schulz loop, derived
in fp64 on the CPU.

TEST INFRASTRUCTURE ONLY, like the rest of oracle/: it produces an input table
(the rows are a runtime input of the Muon step), and shares no code with the
CUDA path.

The pages ("Cara Melatih ChatGPT Sendiri dengan Budget 50 Dolar", section
"2. Pengoptimal Muon (nanochat/optim.py)", coefficient list; its dev.to
translation, section "2. ตัวปรับปรุง Muon") call the per-iteration (a, b, c)
rows "Polar Express", print the first two to three decimals, (8.156, -22.483,
15.879) and (4.043, -2.809, 0.500), and elide the other three.  Polar Express
(Amsel, Persson, Musco and Gower, 2025) builds such a table greedily: the
singular values of the normalised update are known to lie in an interval
[l, u]; each iteration takes the odd quintic p(x) = a x + b x^3 + c x^5 that is
closest to 1 in the max norm on that interval, and the next interval is the
image of the current one under p.  Finite precision adds adjustments to that
plain step.  The pages state none of the construction's parameters; the
readings taken here, each the plainest that reproduces the printed rows, are:

  * start: l_0 = 1e-3 (the smallest singular value, relative to the largest
    after Frobenius normalisation, that the table is built for), u_0 = 1;
  * cushion: the polynomial is fitted on [max(l, u / 50), u], so an iteration
    whose l is tiny is not driven by singular values it cannot move anyway;
  * recentring: the fitted p is scaled by 2 / (p(l) + p(u)), so that the image
    of the true interval [l, u] is centred on 1;
  * safety: x is replaced by x / 1.02 (a / 1.02, b / 1.02^3, c / 1.02^5) in
    every row whose output feeds another row, so that singular values a
    little above u after rounding stay inside the next polynomial's interval;
    the last row feeds none and keeps its output band centred on 1;
  * next interval: l <- p(l) with the final row, u <- 2 - l.

With these, the first two rows come out as (8.15655, -22.48329, 15.87877) and
(4.04293, -2.80892, 0.50002): each printed figure is within one unit of its
last decimal, and all but the first row's leading term (8.15655 printed as
8.156, cut rather than rounded) round to the printed figure.  A plain minimax
on [l_0, 1] with none of the adjustments gives (8.470, -25.108, 18.629)
instead.  The five rows map every x in [1e-3, 1] into [0.8589, 1.1411].

Run ``python -m oracle.polar_express`` to print the table that
tests/golden/polar_express_rows.txt holds.
"""
from __future__ import annotations

import numpy as np

L0 = 1e-3
CUSHION = 1.0 / 50.0
SAFETY = 1.02
ROWS = 5


def quintic(x, abc):
    a, b, c = abc
    x = np.asarray(x, dtype=np.float64)
    return a * x + b * x ** 3 + c * x ** 5


def minimax_odd_quintic(lo: float, hi: float, tol: float = 1e-15, max_iter: int = 200):
    """The odd quintic p minimising max |1 - p(x)| over [lo, hi] (0 < lo <= hi).

    Returns (a, b, c, E) with E the minimal max error.  Remez exchange on the
    four points where the error of the best approximation alternates
    (equioscillation): lo, the two interior critical points of p, and hi,
    with 1 - p = +E, -E, +E, -E there.  When the interval shrinks to a point
    the best polynomial is the one flat to second order at it:
    p(hi) = 1, p'(hi) = p''(hi) = 0, i.e. (15/8, -10/8, 3/8) scaled to hi.
    """
    if not (0.0 < lo <= hi):
        raise ValueError("need 0 < lo <= hi")
    if lo / hi > 1.0 - 1e-7:
        return 15.0 / 8.0 / hi, -10.0 / 8.0 / hi ** 3, 3.0 / 8.0 / hi ** 5, 0.0
    # starting reference points, spread over the interval
    q, r = lo + (hi - lo) / 4.0, lo + 3.0 * (hi - lo) / 4.0
    E_prev = None
    for _ in range(max_iter):
        pts = (lo, q, r, hi)
        M = np.array([[x, x ** 3, x ** 5, (-1.0) ** i] for i, x in enumerate(pts)])
        a, b, c, E = np.linalg.solve(M, np.ones(4))
        # interior critical points: p'(x) = a + 3 b x^2 + 5 c x^4 = 0, a quadratic in x^2
        disc = 9.0 * b * b - 20.0 * a * c
        if c == 0.0 or disc < 0.0:
            raise ArithmeticError("Remez exchange lost its critical points")
        roots2 = (-3.0 * b + np.array([-1.0, 1.0]) * np.sqrt(disc)) / (10.0 * c)
        if np.any(roots2 <= 0.0):
            raise ArithmeticError("Remez exchange lost its critical points")
        q, r = np.sort(np.sqrt(roots2))
        if E_prev is not None and abs(E - E_prev) <= tol:
            break
        E_prev = E
    return float(a), float(b), float(c), float(E)


def polar_express_rows(n_rows: int = ROWS, l0: float = L0, cushion: float = CUSHION, safety: float = SAFETY):
    """The table, row by row (list of (a, b, c)), and the intervals [l, u] each row was built for."""
    lo, hi = float(l0), 1.0
    rows, intervals = [], []
    for _ in range(n_rows):
        intervals.append((lo, hi))
        a, b, c, _ = minimax_odd_quintic(max(lo, cushion * hi), hi)
        k = 2.0 / (quintic(lo, (a, b, c)) + quintic(hi, (a, b, c)))
        sf = safety if len(rows) < n_rows - 1 else 1.0
        row = (a * k / sf, b * k / sf ** 3, c * k / sf ** 5)
        rows.append(row)
        lo = float(quintic(lo, row))
        hi = 2.0 - lo
    return rows, intervals


def main() -> None:
    rows, intervals = polar_express_rows()
    print(f"# Polar Express rows: l0 = {L0}, cushion u/{1.0 / CUSHION:g}, safety {SAFETY} (all rows but the last), "
          f"interval update l <- p(l), u <- 2 - l")
    print("# written by `python -m oracle.polar_express`; columns: a b c, then the interval l u the row was built for")
    for (a, b, c), (lo, hi) in zip(rows, intervals):
        print(f"{float(a)!r} {float(b)!r} {float(c)!r} {float(lo)!r} {float(hi)!r}")


if __name__ == "__main__":
    main()
