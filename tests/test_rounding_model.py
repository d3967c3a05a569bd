"""Where the GPU parity tolerances come from: a rounding model of the CUDA path,
run against the fp64 oracle on the CPU.

The model is not the CUDA code.  It repeats, in numpy, only the points where
the kernels round (bf16 is round-to-nearest-even, accumulation is fp32):

  m' = fp32(beta m + g), u = fp32(g + beta m')        (one fma each)
  X0 = bf16(u), oriented; s = fp32(1 / (||u||_F + eps))
  iteration k with row (a, b, c), s applied in the first iteration only:
    A  = bf16(s^2 fp32(X X^T))
    B' = bf16(fp32(c fp32(A A) + fp32(b A)) + a I)     (a I folded into the polynomial)
    X  = bf16(s fp32(B' X))                            (the last iteration keeps fp32)
  O  = the last X, oriented back

and measures O's relative Frobenius error against oracle.muon_matrix on seeded
inputs of the workloads' distributions.  fp32 accumulation is modelled as an
fp64 product rounded once to fp32; its own error (about 1e-7 per sum) is far
below bf16's unit roundoff 2^-8, which dominates every result here.

What it shows, and the GPU tests use:
  * matrices with both sides >= 64 stay well inside 2e-2 after 5 iterations;
  * one iteration stays inside 5e-3 (the tight check of the ragged-shape test);
  * 8 x 8 matrices reach errors above 2e-2 (the Frobenius error does not
    average over many entries), but stay below 6e-2 over 40 seeded draws, the
    bound the GPU tests give matrices with a side below 64;
  * with the five-row Polar Express table (first row 8.156, -22.483, 15.879)
    sides of 64 and more still stay inside 2e-2, but matrices with a side
    below 64 reach 8e-2 to 9e-2: the large a I and b A terms of its rows
    cancel on bf16 operands, and small matrices do not average the error out.
    The GPU tests give them 1.2e-1 with that table.
"""
import numpy as np
import pytest

import oracle

BETA = np.float32(0.95)
EPS = 1e-7


def bf16(x):
    """Round float32 values to bfloat16 (round to nearest, ties to even); returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    return rounded.view(np.float32)


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def model_o(g, m, coeffs, ns_steps, beta=BETA, eps=EPS):
    """O of one matrix as the kernels round it (float64 array of the stored shape)."""
    g32, m32 = g.astype(np.float32), m.astype(np.float32)
    b = np.float64(beta)
    mn = f32(b * m32.astype(np.float64) + g32)
    u = f32(g32.astype(np.float64) + b * mn.astype(np.float64))
    tall = g.shape[0] > g.shape[1]
    X = bf16(u.T if tall else u).astype(np.float64)
    nrm = np.sqrt(np.sum(u.astype(np.float64) ** 2))
    s = np.float64(f32(1.0 / (nrm + eps)))
    for k in range(ns_steps):
        a, bb, c = (np.float64(np.float32(v)) for v in coeffs[k])
        sk = s if k == 0 else 1.0
        A = bf16(f32(np.float64(f32(sk * sk)) * f32(X @ X.T))).astype(np.float64)
        AA = f32(A @ A).astype(np.float64)
        B = f32(c * AA + f32(bb * A)).astype(np.float64)
        B = bf16(f32(B + a * np.eye(B.shape[0]))).astype(np.float64)
        Y = f32(sk * f32(B @ X)).astype(np.float64)
        X = Y if k == ns_steps - 1 else bf16(Y).astype(np.float64)
    return X.T if tall else X


def model_error(shape, seed, ns_steps=5, coeffs=oracle.DEFAULT_COEFFS):
    """Relative Frobenius error of the model's O against the oracle on one seeded draw
    (g ~ N(0, 1e-3^2) with a per-row factor U[0.5, 2], m ~ N(0, 1e-3^2), as the workloads)."""
    rng = np.random.default_rng(seed)
    r, c = shape
    g = (rng.standard_normal(shape) * 1e-3 * rng.uniform(0.5, 2.0, (r, 1))).astype(np.float32)
    m = (rng.standard_normal(shape) * 1e-3).astype(np.float32)
    p = (rng.standard_normal(shape) / np.sqrt(c)).astype(np.float32)
    _, _, O_ref = oracle.muon_matrix(p, g, m, lr=np.float32(0.02), beta=BETA, nesterov=True,
                                     ns_steps=ns_steps, coeffs=coeffs, eps=EPS)
    O = model_o(g, m, coeffs, ns_steps)
    return np.linalg.norm(O - O_ref) / np.linalg.norm(O_ref)


def test_bf16_rounding_helper():
    # exact on representable values, ties to even, and within 2^-8 relative otherwise (8 significant bits)
    assert bf16(np.float32(1.0)) == 1.0 and bf16(np.float32(-3.0)) == -3.0
    one_ulp = np.float32(2.0 ** -7)                      # bf16 spacing at 1.0
    assert bf16(np.float32(1.0) + one_ulp / 2) == 1.0    # tie: to the even neighbour (1.0)
    assert bf16(np.float32(1.0) + 3 * one_ulp / 2) == np.float32(1.0) + 2 * one_ulp
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32)
    assert np.all(np.abs(bf16(x) - x) <= 2.0 ** -8 * np.abs(x))


def test_model_with_exact_rounding_is_the_oracle():
    # with rounding switched off the model must reduce to the oracle (pins the model's algebra:
    # the folded a I, the scale in the first iteration only, the orientation)
    global bf16
    saved = bf16
    try:
        bf16 = lambda x: np.asarray(x, dtype=np.float32)  # noqa: E731
        for shape in [(24, 40), (40, 24), (16, 16)]:
            assert model_error(shape, 5) < 1e-5, shape
    finally:
        bf16 = saved


@pytest.mark.parametrize("shape", [(128, 128), (512, 128), (128, 512), (264, 264), (136, 200)])
def test_sides_of_64_and_more_stay_well_inside_the_main_bound(shape):
    errs = [model_error(shape, seed) for seed in range(2)]
    assert max(errs) < 1.5e-2, errs


@pytest.mark.parametrize("shape", [(136, 200), (200, 136), (8, 1024), (1024, 8), (264, 264)])
def test_one_iteration_stays_inside_the_tight_bound(shape):
    assert model_error(shape, 11, ns_steps=1) < 3.5e-3


def test_eight_by_eight_needs_the_wider_bound():
    errs = np.array([model_error((8, 8), seed) for seed in range(40)])
    # above the main 2e-2 for some draws, so the main bound would be wrong for such shapes ...
    assert errs.max() > 2e-2
    # ... and below the 6e-2 the GPU tests allow them, with room for the GPU's own summation order
    assert errs.max() < 4.5e-2, float(errs.max())
    assert np.median(errs) < 2.5e-2


def test_polar_express_table_bounds():
    import pretraining_optimizer_step_b300 as mu
    pe = np.array(mu.POLAR_EXPRESS_COEFFS)
    for shape in [(136, 200), (264, 264), (128, 384)]:
        assert model_error(shape, 3, coeffs=pe) < 1.7e-2, shape
    small = np.array([model_error((8, 8), seed, coeffs=pe) for seed in range(60)] +
                     [model_error(s, seed, coeffs=pe) for s in [(8, 1024), (1024, 8)] for seed in range(4)])
    assert small.max() > 6e-2              # the default table's small-side bound would not hold
    assert small.max() < 1.0e-1, float(small.max())   # ... and 1.2e-1 leaves room for the GPU's order
