"""fp64 CPU oracle of the Muon optimizer step and of the AdamW step for the
parameters Muon does not take (ctypes wrapper around muon_oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the product library never
does, and it shares no code with the CUDA path.

The method and the readings taken where the pages are silent are stated in the
header of ``muon_oracle.c``; the sources are the pages "Cara Melatih ChatGPT
Sendiri dengan Budget 50 Dolar" (apidog.com), section "2. Pengoptimal Muon
(nanochat/optim.py)", and its dev.to translation, section "2. ตัวปรับปรุง Muon".
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "muon_oracle.c")
_LIB = os.path.join(_HERE, "libmuon_oracle.so")

# The fixed quintic of the classic Muon write-up, used for every iteration.
# Its five-fold composition maps (0.01, 1] into about [0.68, 1.13], the band
# the method's description quotes; the pages print only two of the five
# per-iteration "Polar Express" rows, so that table cannot be the default.
DEFAULT_ROW = (3.4445, -4.7750, 2.0315)
DEFAULT_COEFFS = np.array([DEFAULT_ROW] * 5, dtype=np.float64)
# The two "Polar Express" rows the pages print (rounded to 3 decimals there),
# section "2. Pengoptimal Muon", coefficient list.
PAGES_POLAR_EXPRESS_ROWS = np.array([(8.156, -22.483, 15.879), (4.043, -2.809, 0.500)],
                                    dtype=np.float64)
DEFAULT_EPS = 1e-7

_lib = None


def build(force: bool = False) -> str:
    """Compile muon_oracle.c into a shared library beside it; returns its path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", _LIB, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


def bind(lib):
    """Declare the C signatures on a loaded oracle library (also used for test mutants)."""
    f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
    f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
    lib.oracle_momentum.argtypes = [ctypes.c_long, f32p, f32p, ctypes.c_double, ctypes.c_int,
                                    ctypes.c_int, f32p, f64p]
    lib.oracle_momentum.restype = None
    lib.oracle_newton_schulz.argtypes = [ctypes.c_int, ctypes.c_int, f64p, ctypes.c_int, f64p]
    lib.oracle_newton_schulz.restype = ctypes.c_int
    lib.oracle_orthogonalize.argtypes = [ctypes.c_int, ctypes.c_int, f64p, ctypes.c_int, f64p,
                                         ctypes.c_double, f64p]
    lib.oracle_orthogonalize.restype = ctypes.c_int
    lib.oracle_muon_matrix.argtypes = [ctypes.c_int, ctypes.c_int, f32p, f32p, f32p,
                                       ctypes.c_double, ctypes.c_double, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, f64p, ctypes.c_double,
                                       f32p, f32p, f64p]
    lib.oracle_muon_matrix.restype = ctypes.c_int
    lib.oracle_frobenius.argtypes = [ctypes.c_long, f64p]
    lib.oracle_frobenius.restype = ctypes.c_double
    lib.oracle_normuon_scale.argtypes = [ctypes.c_int, ctypes.c_int, f64p, f32p, ctypes.c_double, ctypes.c_double]
    lib.oracle_normuon_scale.restype = None
    lib.oracle_normuon_matrix.argtypes = [ctypes.c_int, ctypes.c_int, f32p, f32p, f32p, ctypes.c_double,
                                          ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int, f64p,
                                          ctypes.c_double, f32p, ctypes.c_double, ctypes.c_double, f32p, f32p, f64p]
    lib.oracle_normuon_matrix.restype = ctypes.c_int
    lib.oracle_adamw.argtypes = [ctypes.c_long, f32p, f32p, f32p, f32p, ctypes.c_double, ctypes.c_double,
                                 ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_int]
    lib.oracle_adamw.restype = None
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = bind(ctypes.CDLL(_LIB))
    return _lib


@contextlib.contextmanager
def using_library(path):
    """Route every call in this module to another build of the oracle (a test mutant)."""
    global _lib
    saved = _load()
    _lib = bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def source_path() -> str:
    return _SRC


def _coeffs(coeffs, K):
    c = np.ascontiguousarray(np.asarray(coeffs, dtype=np.float64).reshape(-1, 3))
    if K is None:
        K = c.shape[0]
    if K > c.shape[0]:
        raise ValueError("ns_steps exceeds the coefficient table")
    return np.ascontiguousarray(c[:max(K, 1)].reshape(-1)), K


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def momentum(g, m, beta, nesterov=True, mode=0):
    """m' (float32) and u (float64) for one matrix; see muon_oracle.c."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    m = np.ascontiguousarray(m, dtype=np.float32)
    m_out = np.empty_like(m)
    u = np.empty(g.shape, dtype=np.float64)
    _load().oracle_momentum(g.size, g, m, float(beta), int(bool(nesterov)), int(mode), m_out, u)
    return m_out, u


def newton_schulz(X, coeffs=DEFAULT_COEFFS, ns_steps=None):
    """The quintic loop on an oriented, normalised X (copied; returns the result)."""
    X = np.array(X, dtype=np.float64, order="C", copy=True)
    c, K = _coeffs(coeffs, ns_steps)
    if _load().oracle_newton_schulz(X.shape[0], X.shape[1], X, K, c) != 0:
        raise MemoryError("oracle allocation failed")
    return X


def orthogonalize(u, coeffs=DEFAULT_COEFFS, ns_steps=None, eps=DEFAULT_EPS):
    """O for one stored r x c direction u: orient, normalise, iterate, orient back."""
    u = np.ascontiguousarray(u, dtype=np.float64)
    r, cc = u.shape
    O = np.empty((r, cc), dtype=np.float64)
    c, K = _coeffs(coeffs, ns_steps)
    if _load().oracle_orthogonalize(r, cc, u, K, c, float(eps), O) != 0:
        raise MemoryError("oracle allocation failed")
    return O


def muon_matrix(p, g, m, lr, beta, nesterov=True, ns_steps=None, coeffs=DEFAULT_COEFFS,
                eps=DEFAULT_EPS, mode=0):
    """One Muon step on one stored matrix: returns (p' float32, m' float32, O float64)."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    g = np.ascontiguousarray(g, dtype=np.float32)
    m = np.ascontiguousarray(m, dtype=np.float32)
    r, cc = p.shape
    c, K = _coeffs(coeffs, ns_steps)
    p_out = np.empty_like(p)
    m_out = np.empty_like(m)
    O = np.empty((r, cc), dtype=np.float64)
    rc = _load().oracle_muon_matrix(r, cc, p, g, m, float(lr), float(beta), int(bool(nesterov)),
                                    int(mode), K, c, float(eps), p_out, m_out, O)
    if rc != 0:
        raise MemoryError("oracle allocation failed")
    return p_out, m_out, O


def adamw(p, g, m, v, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step=1):
    """One AdamW step on one tensor (copies in, returns (p', m', v') as float32 arrays)."""
    p = np.array(p, dtype=np.float32, order="C", copy=True)
    m = np.array(m, dtype=np.float32, order="C", copy=True)
    v = np.array(v, dtype=np.float32, order="C", copy=True)
    g = np.ascontiguousarray(g, dtype=np.float32)
    if int(step) < 1:
        raise ValueError("step counts from 1")
    _load().oracle_adamw(p.size, p.reshape(-1), g.reshape(-1), m.reshape(-1), v.reshape(-1), float(lr),
                         float(beta1), float(beta2), float(eps), float(weight_decay), int(step))
    return p, m, v


NORMUON_BETA2 = 0.95
NORMUON_EPS = 1e-10


def normuon_scale(O, V, beta2=NORMUON_BETA2, eps=NORMUON_EPS):
    """NorMuon-scaled copy of O (stored r x c) and the updated per-row state V (float32)."""
    O = np.array(O, dtype=np.float64, order="C", copy=True)
    V = np.array(V, dtype=np.float32, order="C", copy=True).reshape(-1)
    r, c = O.shape
    if V.size != r:
        raise ValueError("V holds one value per stored row")
    _load().oracle_normuon_scale(r, c, O, V, float(beta2), float(eps))
    return O, V


def normuon_matrix(p, g, m, V, lr, beta, nesterov=True, ns_steps=None, coeffs=DEFAULT_COEFFS, eps=DEFAULT_EPS,
                   mode=0, beta2=NORMUON_BETA2, eps2=NORMUON_EPS):
    """One Muon step with NorMuon scaling: returns (p', m', V', O')."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    g = np.ascontiguousarray(g, dtype=np.float32)
    m = np.ascontiguousarray(m, dtype=np.float32)
    V = np.array(V, dtype=np.float32, order="C", copy=True).reshape(-1)
    r, cc = p.shape
    c, K = _coeffs(coeffs, ns_steps)
    p_out = np.empty_like(p)
    m_out = np.empty_like(m)
    O = np.empty((r, cc), dtype=np.float64)
    rc = _load().oracle_normuon_matrix(r, cc, p, g, m, float(lr), float(beta), int(bool(nesterov)), int(mode), K,
                                       c, float(eps), V, float(beta2), float(eps2), p_out, m_out, O)
    if rc != 0:
        raise MemoryError("oracle allocation failed")
    return p_out, m_out, V, O
