"""The seeded input generators: shapes and distributions of the workloads."""
import math

import numpy as np
import pytest
import torch

import workloads


def test_stack_shapes_follow_width_64_depth():
    for name, depth in workloads.STACK_DEPTHS.items():
        shapes = workloads.config_shapes(name)
        d = 64 * depth
        assert len(shapes) == 6 * depth
        assert shapes[:6] == [(d, d)] * 4 + [(4 * d, d), (d, 4 * d)]
    assert sum(r * c for r, c in workloads.config_shapes("d26")) == 863_895_552
    assert sum(r * c for r, c in workloads.config_shapes("d12")) == 84_934_656


def test_sweep_shapes():
    assert workloads.config_shapes("sweep_512_tall") == [(2048, 512)] * 64
    assert workloads.config_shapes("sweep_512_wide") == [(512, 2048)] * 64
    assert len(workloads.sweep_names()) == 18


def test_generators_are_deterministic_and_distinct():
    a = workloads.make_stack("d2", "cpu", seed=0)
    b = workloads.make_stack("d2", "cpu", seed=0)
    for x, y in zip(a[0] + a[1] + a[2], b[0] + b[1] + b[2]):
        assert torch.equal(x, y)
    c = workloads.make_stack("d2", "cpu", seed=1)
    assert not torch.equal(a[1][0], c[1][0])
    g1 = workloads.make_grad("d2", 0, (128, 128), "cpu", 0, step=1)
    assert not torch.equal(a[1][0], g1)
    assert len({workloads.tensor_seed(0, "d2", i, k) for i in range(12) for k in "pgm"}) == 36


def test_distributions():
    p, g, m, shapes = workloads.make_stack("d12", "cpu", indices=[4])
    r, c = shapes[0]
    assert abs(p[0].std().item() * math.sqrt(c) - 1.0) < 0.01
    assert abs(m[0].std().item() / 1e-3 - 1.0) < 0.01
    # per-row factor U[0.5, 2]: row RMS / 1e-3 spans about [0.5, 2]
    rms = g[0].pow(2).mean(dim=1).sqrt() / 1e-3
    assert 0.45 < rms.min().item() < 0.6 and 1.9 < rms.max().item() < 2.1


def test_sweep_rank_deficient_mix():
    name = "sweep_256_tall"
    g0 = workloads.make_grad(name, 0, (1024, 256), "cpu").double().numpy()
    g1 = workloads.make_grad(name, 1, (1024, 256), "cpu").double().numpy()
    s0 = np.linalg.svd(g0, compute_uv=False)
    s1 = np.linalg.svd(g1, compute_uv=False)
    rank = 256 // 8
    assert s0[rank] / s0[0] < 1e-3          # rank min/8 plus 1e-6 noise
    assert s0[rank - 1] / s0[0] > 1e-2
    assert s1[-1] / s1[0] > 0.1             # full rank
    assert abs(g1.std() / 1e-3 - 1) < 0.02
