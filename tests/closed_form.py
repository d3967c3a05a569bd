"""The Muon update O in closed form, for checking the GPU at sizes the fp64
oracle cannot finish in a test.

Every Newton-Schulz step X <- a X + b (X X^T) X + c (X X^T)^2 X is a polynomial
in X X^T applied to X, so the K steps give O = q(X0 X0^T) X0 with q a matrix
function: if X0 X0^T = U diag(lambda) U^T and x = sqrt(lambda) are the singular
values of X0, each step maps x to x f(x) with f(x) = a + b x^2 + c x^4, and q
takes the product of those factors.  The momentum, the normalisation and the
orientation are those of the method (SGD-Nesterov form, X0 = u / (||u||_F +
eps), wide side as columns).  numpy fp64; eigh of the m x m Gram matrix.
"""
import numpy as np


def closed_form_o(g, m, beta, coeffs, eps=1e-7, nesterov=True):
    r, c = g.shape
    g = np.asarray(g, dtype=np.float64)
    bf = float(np.float32(beta))
    m1 = bf * np.asarray(m, dtype=np.float64) + g
    u = g + bf * m1 if nesterov else m1
    X = u.T if r > c else u
    X = X / (np.linalg.norm(u) + eps)
    lam, U = np.linalg.eigh(X @ X.T)
    x = np.sqrt(np.clip(lam, 0.0, None))
    s = np.ones_like(x)
    for a, b, cc in coeffs:
        f = a + b * x * x + cc * x ** 4
        s *= f
        x = x * f
    O = (U * s) @ (U.T @ X)
    return O.T if r > c else O
