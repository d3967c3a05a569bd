"""Helpers of the GPU parity tests: run the CUDA path through the C ABI on seeded
inputs, run the oracle on the same inputs, compare within the stated tolerances.

The step is run as a caller runs it (debug_flags = 0: no debug copy of O, the
launch configuration the benchmark times).  O is recovered from the weight
change: the library applies p' = p - sc O with sc = fp32(lr * sqrt(max(1, r/c))),
so O = (p - p') / sc up to the float32 rounding of p', at most 2^-24 |p'| / sc per
entry: below 1e-5 relative on every workload shape once the iterations have run
(||O||_F is then about sqrt(min side)), a few 1e-5 at ns_steps = 0 (||O||_F = 1).
O is then held to the same bounds as a directly copied O.

Tolerances (per matrix, relative Frobenius): the Newton-Schulz output O within
2e-2, the updated fp32 weights p' within 1e-3, the weight change p' - p within
2e-2; the momentum buffer m' within float32 rounding of its terms; ||u||_F
within 1e-5.  The kernels hold X, A, B in bfloat16 (8 significant bits, unit
roundoff 2^-8) with fp32 accumulation: rounding X0 alone gives O errors of
about 1.7e-3, and five iterations of the default table amplify that to about
1.2e-2 on the workload shapes.  Two cases need wider, derived bounds (see the
tests that use them): matrices with fewer than 64 rows or columns, whose
Frobenius error does not average over many elements, and coefficient rows with
large leading terms such as the pages' (8.156, -22.483, 15.879).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import pretraining_optimizer_step_b300 as mu

TOL_O = 2e-2
TOL_P = 1e-3
TOL_DP = 2e-2


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / nb if nb > 0 else np.linalg.norm(a - b)


def f32(x: float) -> float:
    return float(np.float32(x))


def update_scale(lr, shape):
    """The fp32 factor the library multiplies O by: fp32(lr) * fp32(sqrt(max(1, rows/cols)))."""
    r, c = shape
    return np.float32(np.float32(lr) * np.float32(np.sqrt(max(1.0, r / c))))


def o_from_update(p0, p1, lr, shape):
    """O of one matrix recovered from its weight change (float64)."""
    return (np.asarray(p0, np.float64) - np.asarray(p1, np.float64)) / float(update_scale(lr, shape))


def run_gpu_step(params, grads, moms, lr=0.02, beta=0.95, nesterov=True, ns_steps=5, keep_o=False,
                 stream=None):
    """One step on device tensors (updated in place).  With keep_o (a context made with
    MUON_DEBUG_KEEP_O) returns the debug copies of O (CPU, float32), else []."""
    mu.muon_step(params, grads, moms, lr=lr, beta=beta, nesterov=nesterov, ns_steps=ns_steps,
                 stream=stream)
    mu.muon_get_status(stream)
    outs = []
    if keep_o:
        for i, p in enumerate(params):
            o = torch.empty_like(p)
            mu.muon_debug_copy_ns_output(i, o, stream)
            outs.append(o)
        torch.cuda.synchronize()
        outs = [o.cpu().numpy() for o in outs]
    return outs


def check_momentum(i, g0, m0, m1, m_ref, beta):
    """m' against the oracle's.  The GPU forms m' with one fma (mode 0: a single rounding) or a
    rounded product (1-beta) g and an fma (mode 1: two roundings), so the error is bounded by
    float32 ulps of the terms, not of the (possibly cancelled) result."""
    bf = f32(beta)
    terms = np.abs(bf * m0.astype(np.float64)) + np.abs(g0.astype(np.float64))
    err = np.abs(m1.astype(np.float64) - m_ref.astype(np.float64))
    bound = 2.5e-7 * np.abs(m_ref.astype(np.float64)) + 1.2e-7 * terms
    assert np.all(err <= bound), (i, "m'", float(np.max(err - bound)))


def check_matrix(i, p0, g0, m0, p1, m1, O_gpu, lr, beta, nesterov, ns_steps, coeffs, eps=1e-7,
                 mode=0, norm_gpu=None, tol_o=TOL_O):
    """Compare one matrix's GPU results with the oracle run on the same inputs.  O_gpu None:
    O is recovered from the weight change."""
    if O_gpu is None:
        O_gpu = o_from_update(p0, p1, lr, p0.shape)
    p_ref, m_ref, O_ref = oracle.muon_matrix(p0, g0, m0, lr=f32(lr), beta=f32(beta), nesterov=nesterov,
                                             ns_steps=ns_steps, coeffs=coeffs, eps=eps, mode=mode)
    report = {}
    check_momentum(i, g0, m0, m1, m_ref, beta)
    if norm_gpu is not None:
        _, u = oracle.momentum(g0, m0, f32(beta), nesterov, mode)
        nrm = float(np.linalg.norm(u))
        assert abs(norm_gpu - nrm) <= 1e-5 * nrm + 1e-30, (i, norm_gpu, nrm)
    if O_gpu is not None:
        if np.linalg.norm(O_ref) == 0:
            assert np.all(O_gpu == 0), i
        else:
            report["O"] = rel_fro(O_gpu, O_ref)
            assert report["O"] <= tol_o, (i, report)
    # p' - p = -lr s O, so a wider bound on O widens those on p' and p' - p alike
    widen = max(1.0, tol_o / TOL_O)
    report["p"] = rel_fro(p1, p_ref)
    assert report["p"] <= TOL_P * widen, (i, report)
    dp_ref = p_ref.astype(np.float64) - p0
    if np.linalg.norm(dp_ref) > 0:
        report["dp"] = rel_fro(p1.astype(np.float64) - p0, dp_ref)
        assert report["dp"] <= TOL_DP * widen, (i, report)
    return report, (p_ref, m_ref)
