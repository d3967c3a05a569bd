"""Parity of the CUDA AdamW step (through the C ABI) with the fp64 oracle.

The kernel computes in fp32, so each result is compared with the oracle within
the rounding of its own formula: m' and v' within a few ulps of their terms;
p' within 2 ulps of the decayed weight, plus 2e-6 of the update, plus the
propagated rounding of m' (a cancellation of b1 m and (1 - b1) g can make m'
much smaller than its terms).  A CPU emulation of the kernel's operation order
stays below half of this bound on 2e6 random elements with forced cancellations.
"""
import numpy as np
import pytest
import torch

import oracle
import pretraining_optimizer_step_b300 as mu
import workloads

pytestmark = pytest.mark.gpu

HP = dict(lr=3e-3, beta1=0.8, beta2=0.95, eps=1e-8, weight_decay=0.05)


def check_tensor(i, p0, g0, m0, v0, p1, m1, v1, step, hp):
    # the C ABI takes the hyperparameters as float32: the oracle gets those exact values
    hp = {k: float(np.float32(v)) for k, v in hp.items()}
    p_ref, m_ref, v_ref = oracle.adamw(p0, g0, m0, v0, step=step, **hp)
    b1, b2 = np.float32(hp["beta1"]), np.float32(hp["beta2"])
    g64 = g0.astype(np.float64)
    # m' and v': one fma of two terms, each term's rounding bounded by its size
    m_terms = np.abs(b1 * m0.astype(np.float64)) + np.abs((1 - b1) * g64)
    v_terms = np.abs(b2 * v0.astype(np.float64)) + np.abs((1 - b2) * g64 * g64)
    assert np.all(np.abs(m1 - m_ref.astype(np.float64)) <= 2.5e-7 * m_terms + 1e-38), (i, "m")
    assert np.all(np.abs(v1 - v_ref.astype(np.float64)) <= 5e-7 * v_terms + 1e-38), (i, "v")
    bc1 = 1 - hp["beta1"] ** step
    bc2 = 1 - hp["beta2"] ** step
    ss = hp["lr"] / bc1
    den = np.sqrt(v_ref.astype(np.float64) / bc2) + hp["eps"]
    upd = ss * m_ref.astype(np.float64) / den
    # the decayed weight and the update are each rounded in fp32; m' can be a cancellation of
    # its two terms, so its absolute rounding (scaled by ss / den) is bounded by those terms
    pdec = np.abs(p0.astype(np.float64) * (1 - hp["lr"] * hp["weight_decay"]))
    bound = 2.4e-7 * pdec + 2e-6 * np.abs(upd) + 3e-7 * ss * m_terms / den + 1e-37
    err = np.abs(p1.astype(np.float64) - p_ref.astype(np.float64))
    assert np.all(err <= bound), (i, "p", float(np.max(err / bound)))
    return p_ref, m_ref, v_ref


def run_steps(numels, steps=3, hp=HP, seed=3):
    """Several steps on device state carried from step to step; each step is checked against
    the oracle run on the device's own state from before that step."""
    rng = np.random.default_rng(seed)
    dev = []
    for n in numels:
        p = (rng.standard_normal(n) * 0.02).astype(np.float32)
        m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        v = ((rng.standard_normal(n) * 1e-3) ** 2).astype(np.float32)
        dev.append([torch.tensor(x, device="cuda") for x in (p, m, v)])
    for step in range(1, steps + 1):
        before = [[x.cpu().numpy().copy() for x in d] for d in dev]
        gs = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for n in numels]
        dg = [torch.tensor(g, device="cuda") for g in gs]
        mu.muon_adamw_step([d[0] for d in dev], dg, [d[1] for d in dev], [d[2] for d in dev], step=step, **hp)
        torch.cuda.synchronize()
        for i in range(len(numels)):
            p0, m0, v0 = before[i]
            p1, m1, v1 = (dev[i][k].cpu().numpy() for k in range(3))
            check_tensor(i, p0, gs[i], m0, v0, p1, m1, v1, step, hp)


def test_ragged_tensor_list_three_steps():
    # tails of 1-3 elements, chunk boundaries (16384), single scalars
    run_steps([1, 3, 5, 8, 1000, 4097, 16384, 16387, 40000], steps=3)


def test_many_tensors_span_several_launches():
    # more than 128 tensors: the host splits them over launches
    run_steps([7 + (i % 13) * 4 for i in range(300)], steps=2, seed=4)


def test_zero_weight_decay_and_large_eps():
    run_steps([4096, 33], steps=2, hp=dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-3, weight_decay=0.0), seed=5)


@pytest.mark.parametrize("name", ["d12", "d26"])
def test_adamw_set_sampled(name):
    # d26's set is the one the benchmark's AdamW leg times
    p, g, m, v, shapes = workloads.make_adamw_set(name, "cuda")
    host = [[t.cpu().numpy().reshape(-1).copy() for t in (p[i], g[i], m[i], v[i])] for i in range(len(p))]
    mu.muon_adamw_step(p, g, m, v, step=7, **HP)
    torch.cuda.synchronize()
    for i in (0, 1, 2, len(p) - 2, len(p) - 1):
        p0, g0, m0, v0 = host[i]
        sel = slice(None) if p0.size < 100000 else slice(0, p0.size, 97)   # a strided sample of the big tables
        p1 = p[i].reshape(-1).cpu().numpy()[sel]
        m1 = m[i].reshape(-1).cpu().numpy()[sel]
        v1 = v[i].reshape(-1).cpu().numpy()[sel]
        check_tensor(i, p0[sel], g0[sel], m0[sel], v0[sel], p1, m1, v1, 7, HP)


def test_argument_errors_enqueue_nothing():
    t = [torch.ones(64, device="cuda") for _ in range(4)]
    before = [x.clone() for x in t]
    ok = mu.AdamWArgs([t[0]], [t[1]], [t[2]], [t[3]])
    assert mu.muon_adamw_step(ok, step=0, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_adamw_step(ok, beta1=1.0, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_adamw_step(ok, beta2=-0.1, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_adamw_step(ok, eps=-1.0, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_adamw_step(ok, lr=float("nan"), check=False) == mu.MUON_ERR_INVALID_ARG
    bad = mu.AdamWArgs([t[0].data_ptr() + 4], [t[1]], [t[2]], [t[3]], numels=[60])
    assert mu.muon_adamw_step(bad, check=False) == mu.MUON_ERR_MISALIGNED
    assert mu.muon_adamw_step([], [], [], [], check=False) == mu.MUON_OK
    # a zero-size tensor is skipped, even with a null pointer
    z = mu.AdamWArgs([0], [0], [0], [0], numels=[0])
    assert mu.muon_adamw_step(z, check=False) == mu.MUON_OK
    torch.cuda.synchronize()
    for a, b in zip(before, t):
        assert torch.equal(a, b)
