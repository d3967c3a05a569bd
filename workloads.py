"""Seeded synthetic inputs for the Muon step: parameter stacks shaped like the
depth-parameterised nanochat models, and the square / 4:1 shape sweep.

This module only draws random numbers and lists shapes; it holds none of the
method's arithmetic, and both the oracle-side tests and the CUDA-side tests and
bench draw their inputs from it.

Stacks (width = 64 * depth): per layer four d x d attention matrices
(q, k, v, output projection), the MLP input 4d x d and the MLP output d x 4d,
stored as PyTorch (out_features, in_features).  Distributions:
  p ~ N(0, 1/cols); g ~ N(0, 1e-3^2) times a per-row factor U[0.5, 2];
  m ~ N(0, 1e-3^2).  Seed 0.  Later steps draw fresh gradients (the step index
  is part of the seed); params and momentum carry over.
Sweep: 64 matrices of one shape; g std 1e-3; every even-indexed matrix is rank
min(rows, cols)/8, g = L R * 1e-3 / sqrt(rank) + 1e-6 N(0, 1), no row factor.
"""
from __future__ import annotations

import math

import torch

STACK_DEPTHS = {"d2": 2, "d12": 12, "d20": 20, "d26": 26}
SWEEP_SIZES = (256, 512, 1024, 2048, 4096, 8192)
SWEEP_COUNT = 64
HYPER = {"lr": 0.02, "beta": 0.95, "nesterov": True, "ns_steps": 5}

_MASK = (1 << 64) - 1


def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _MASK
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def tensor_seed(seed: int, config: str, mat: int, kind: str, step: int = 0) -> int:
    """A 63-bit seed for one tensor, mixed from its identity."""
    h = _splitmix64(seed)
    for part in (sum(ord(ch) * 131 ** i for i, ch in enumerate(config)) & _MASK, mat,
                 {"p": 1, "g": 2, "m": 3, "L": 4, "R": 5, "n": 6, "s": 7}[kind], step):
        h = _splitmix64(h ^ (part & _MASK))
    return h & ((1 << 63) - 1)


def layer_shapes(dim: int):
    return [(dim, dim)] * 4 + [(4 * dim, dim), (dim, 4 * dim)]


def config_shapes(name: str):
    """Stored (rows, cols) of every matrix of a named workload.

    "dNxL" is the first L layers of the dN stack (same shapes, fewer matrices),
    used to profile a stack's kernels on a small footprint."""
    if name in STACK_DEPTHS:
        depth = STACK_DEPTHS[name]
        return layer_shapes(64 * depth) * depth
    if name.startswith("d") and "x" in name and name.split("x")[0] in STACK_DEPTHS:
        base, layers = name.split("x")
        return layer_shapes(64 * STACK_DEPTHS[base]) * int(layers)
    if name.startswith("sweep_"):
        _, n, kind = name.split("_")
        n = int(n)
        shape = {"sq": (n, n), "tall": (4 * n, n), "wide": (n, 4 * n)}[kind]
        return [shape] * SWEEP_COUNT
    raise KeyError(name)


def sweep_names():
    return [f"sweep_{n}_{k}" for n in SWEEP_SIZES for k in ("sq", "tall", "wide")]


def _gen(device, s: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def _normal(shape, std, device, s):
    return torch.randn(shape, generator=_gen(device, s), device=device, dtype=torch.float32) * std


def make_param(name: str, i: int, shape, device, seed: int = 0):
    return _normal(shape, 1.0 / math.sqrt(shape[1]), device, tensor_seed(seed, name, i, "p"))


def make_momentum(name: str, i: int, shape, device, seed: int = 0):
    return _normal(shape, 1e-3, device, tensor_seed(seed, name, i, "m"))


def make_grad(name: str, i: int, shape, device, seed: int = 0, step: int = 0):
    rows, cols = shape
    if name.startswith("sweep_"):
        if i % 2 == 0:
            rank = max(1, min(rows, cols) // 8)
            L = _normal((rows, rank), 1.0, device, tensor_seed(seed, name, i, "L", step))
            R = _normal((rank, cols), 1.0, device, tensor_seed(seed, name, i, "R", step))
            noise = _normal(shape, 1e-6, device, tensor_seed(seed, name, i, "n", step))
            return (L @ R) * (1e-3 / math.sqrt(rank)) + noise
        return _normal(shape, 1e-3, device, tensor_seed(seed, name, i, "g", step))
    g = _normal(shape, 1e-3, device, tensor_seed(seed, name, i, "g", step))
    scale = torch.rand((rows, 1), generator=_gen(device, tensor_seed(seed, name, i, "s", step)),
                       device=device, dtype=torch.float32) * 1.5 + 0.5
    return g * scale


def make_stack(name: str, device="cpu", seed: int = 0, indices=None):
    """(params, grads, momenta, shapes) for a workload, optionally a subset of its matrices."""
    shapes = config_shapes(name)
    idx = range(len(shapes)) if indices is None else indices
    params = [make_param(name, i, shapes[i], device, seed) for i in idx]
    grads = [make_grad(name, i, shapes[i], device, seed, 0) for i in idx]
    moms = [make_momentum(name, i, shapes[i], device, seed) for i in idx]
    return params, grads, moms, [shapes[i] for i in idx]


VOCAB = 32768  # the tokenizer's vocabulary size


def adamw_shapes(name: str):
    """The parameters a dN model sends to AdamW (the optimizer split): the token embedding and
    the untied lm_head (vocab x d each), two scalar lambdas per layer, the 24-wide smear gate
    and the backout lambda."""
    depth = STACK_DEPTHS[name]
    d = 64 * depth
    return [(VOCAB, d), (VOCAB, d)] + [(1,)] * (2 * depth) + [(24,), (1,)]


def make_adamw_set(name: str, device="cpu", seed: int = 0):
    """(params, grads, exp_avg, exp_avg_sq, shapes) for the AdamW parameters of a dN model:
    p ~ N(0, 0.02^2), g ~ N(0, 1e-3^2), exp_avg ~ N(0, 1e-3^2), exp_avg_sq = N(0, 1e-3^2)^2."""
    shapes = adamw_shapes(name)
    tag = name + "_adamw"
    ps = [_normal(s, 0.02, device, tensor_seed(seed, tag, i, "p")) for i, s in enumerate(shapes)]
    gs = [_normal(s, 1e-3, device, tensor_seed(seed, tag, i, "g")) for i, s in enumerate(shapes)]
    ms = [_normal(s, 1e-3, device, tensor_seed(seed, tag, i, "m")) for i, s in enumerate(shapes)]
    vs = [_normal(s, 1e-3, device, tensor_seed(seed, tag, i, "s")) ** 2 for i, s in enumerate(shapes)]
    return ps, gs, ms, vs, shapes


def make_custom(shapes, device="cpu", seed: int = 0, tag: str = "custom"):
    """Stack-style inputs for an arbitrary list of shapes (tests of edge cases)."""
    params = [make_param(tag, i, s, device, seed) for i, s in enumerate(shapes)]
    grads = [make_grad(tag, i, s, device, seed, 0) for i, s in enumerate(shapes)]
    moms = [make_momentum(tag, i, s, device, seed) for i, s in enumerate(shapes)]
    return params, grads, moms, list(shapes)
