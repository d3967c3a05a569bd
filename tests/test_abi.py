"""The C ABI on the CPU: libmuon.so loads, exports every function include/muon.h
declares, validates arguments, and its host-only planner counts work the way
the tiling defines it (checked against an independent enumeration here)."""
import ctypes
import os
import math

import pytest
import torch

import pretraining_optimizer_step_b300 as mu
import workloads


@pytest.fixture(scope="module")
def L():
    return mu.lib()


def test_library_exports_every_declared_symbol(L):
    names = mu.declared_symbols()
    assert len(names) >= 10
    raw = ctypes.CDLL(mu.LIB_PATH)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing


def test_library_hides_internal_symbols():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", mu.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(mu.declared_symbols()) <= exported
    assert not [s for s in exported if "launch_ns_pair" in s or "compute_layout" in s]


def test_status_strings(L):
    for code in range(0, 11):
        s = mu.muon_status_string(code)
        assert s and s != "unknown status"
    assert mu.muon_status_string(1234) == "unknown status"


def test_step_before_init_is_rejected(L):
    mu.muon_destroy()
    args = mu.StepArgs([16], [16], [16], shapes=[(8, 8)])
    assert mu.muon_step(args, check=False) == mu.MUON_ERR_NOT_INITIALIZED
    assert mu.muon_get_status(check=False) == mu.MUON_ERR_NOT_INITIALIZED
    assert mu.lib().muon_get_step_info(None) == mu.MUON_ERR_NOT_INITIALIZED


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_init_without_gpu_reports_unsupported_device(L):
    assert mu.muon_init(check=False) == mu.MUON_ERR_UNSUPPORTED_DEVICE


def test_init_rejects_bad_configs_before_touching_the_device(L):
    assert mu.muon_init(momentum_mode=7, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_init(coeffs=[(1.0, float("nan"), 0.0)], check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_init(coeffs=[(1.0, 0.0, 0.0)] * 17, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_init(eps=float("inf"), check=False) == mu.MUON_ERR_INVALID_ARG
    cfg = mu.muon_config()
    cfg.coeffs = (ctypes.c_double * 3)(1.0, 0.0, 0.0)
    cfg.n_coeff_rows = 0
    assert L.muon_init(ctypes.byref(cfg)) == mu.MUON_ERR_INVALID_ARG


# ------------------------------------------------------------------ host planner
def enumerate_pair_tiles(m, n):
    """Brute-force tile sets of the CTA-pair tiling (two 128-row blocks per tile).

    Gram/polynomial, rb = number of 128-row blocks: for column step q and row pair
    rp <= q, with rb even the tile is row blocks 2rp, 2rp+1 x column blocks 2q,
    2q+1 (the lower block of a diagonal tile is computed but not stored); with rb
    odd it is row blocks 2rp, 2rp+1 x column blocks 2q-1, 2q for rp < q, and the
    diagonal block 2rp alone (128 x 128) for rp = q.  Every 128 x 128 block on or
    above the diagonal must be stored by exactly one tile.  Axpy: tile (rp, ct) =
    row blocks 2rp, 2rp+1 x 256 columns from 256 ct (128 when fewer than 129
    remain); a tile whose second row block does not exist computes 128 rows
    (M = 128), every other 256.  Returns tile counts and the executed flops per
    unit K (2 x rows x N per tile)."""
    rb = math.ceil(m / 128)
    sym, sym_f = [], 0
    stored = set()
    for q in range(math.ceil(rb / 2)):
        for rp in range(q + 1):
            sym.append((rp, q))
            if rb % 2 == 0:
                rows, cols = (2 * rp, 2 * rp + 1), (2 * q, 2 * q + 1)
            elif rp < q:
                rows, cols = (2 * rp, 2 * rp + 1), (2 * q - 1, 2 * q)
            else:
                rows, cols = (2 * rp,), (2 * rp,)
            assert all(i < rb for i in rows) and all(c < rb for c in cols)
            sym_f += 2 * 128 * len(rows) * 128 * len(cols)
            for i in rows:
                for c in cols:
                    if i <= c:
                        assert (i, c) not in stored
                        stored.add((i, c))
                    else:
                        assert rb % 2 == 0 and rp == q  # only the even-count diagonal tile computes a lower block
    assert stored == {(i, j) for i in range(rb) for j in range(i, rb)}
    axpy, axpy_f = 0, 0
    for rp in range(math.ceil(rb / 2)):
        rows = 256 if 2 * rp + 1 < rb else 128
        for c0 in range(0, n, 256):
            axpy += 1
            axpy_f += 2 * rows * (256 if n - c0 > 128 else 128)
    return len(sym), axpy, sym_f, axpy_f


def expected_plan(shapes, K):
    classes = {}
    for r, c in shapes:
        key = (min(r, c), max(r, c), r > c)
        classes[key] = classes.get(key, 0) + 1
    alg = exe = 0.0
    sym = axpy = 0
    for (m, n, _), G in classes.items():
        s, a, sym_f, axpy_f = enumerate_pair_tiles(m, n)
        sym += G * s
        axpy += G * a
        alg += G * K * (3 * m * m * n + m ** 3)
        exe += G * K * (sym_f * n + sym_f * m + axpy_f * m)   # Gram K = n, polynomial K = m, axpy K = m
    ctas = sum(math.ceil(r / 64) * math.ceil(c / 64) for r, c in shapes)
    elem = sum(22 * r * c for r, c in shapes)
    return len(classes), alg, exe, sym, axpy, ctas, elem


@pytest.mark.parametrize("name", ["d2", "d12", "d20", "d26", "sweep_1024_tall", "sweep_256_sq"])
def test_plan_query_counts(L, name):
    shapes = workloads.config_shapes(name)
    q = mu.muon_plan_query(shapes, ns_steps=5)
    ncls, alg, exe, sym, axpy, ctas, elem = expected_plan(shapes, 5)
    assert q["n_classes"] == ncls
    assert q["ns_alg_flops"] == pytest.approx(alg, rel=1e-12)
    assert q["ns_executed_flops"] == pytest.approx(exe, rel=1e-12)
    assert q["sym_tiles"] == sym and q["axpy_tiles"] == axpy
    assert q["momentum_ctas"] == ctas
    assert q["elementwise_alg_bytes"] == pytest.approx(elem, rel=1e-12)
    assert q["launches"] == 1 + 3 * 5 * math.ceil(ncls / 8)
    ws_min = sum(2 * (2 * min(r, c) * max(r, c) + 2 * min(r, c) ** 2) for r, c in shapes)
    assert q["workspace_bytes"] >= ws_min


def test_plan_query_d26_headline_numbers(L):
    q = mu.muon_plan_query(workloads.config_shapes("d26"), ns_steps=5)
    assert q["n_classes"] == 3                     # square, tall (transposed), wide
    assert q["ns_alg_flops"] == pytest.approx(2.516e13, rel=1e-3)
    assert q["elementwise_alg_bytes"] == pytest.approx(1.90e10, rel=1e-2)
    assert 1.0 < q["ns_executed_flops"] / q["ns_alg_flops"] < 1.3


def test_plan_query_validation(L):
    assert mu.muon_plan_query([(7, 8)], check=False) == mu.MUON_ERR_UNSUPPORTED_SHAPE
    assert mu.muon_plan_query([(12, 16)], check=False) == mu.MUON_ERR_UNSUPPORTED_SHAPE
    assert mu.muon_plan_query([(8, 0)], check=False) == mu.MUON_ERR_UNSUPPORTED_SHAPE
    assert mu.muon_plan_query([(8, 65544)], check=False) == mu.MUON_ERR_UNSUPPORTED_SHAPE
    assert mu.muon_plan_query([(8, 8)], ns_steps=-1, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_plan_query([(8, 8)], ns_steps=17, check=False) == mu.MUON_ERR_INVALID_ARG
    info = mu.muon_plan_info()
    assert L.muon_plan_query(None, -1, 5, ctypes.byref(info)) == mu.MUON_ERR_INVALID_ARG
    assert L.muon_plan_query(None, 1, 5, ctypes.byref(info)) == mu.MUON_ERR_INVALID_ARG
    q = mu.muon_plan_query([], ns_steps=5)
    assert q["launches"] == 0 and q["workspace_bytes"] == 0


def test_plan_query_ns0_and_class_limit(L):
    q = mu.muon_plan_query([(64, 64)], ns_steps=0)
    assert q["launches"] == 2 and q["ns_alg_flops"] == 0
    # nine distinct shape classes need two launch groups per mode
    shapes = [(8 * (k + 1), 64) for k in range(9)]
    q = mu.muon_plan_query(shapes, ns_steps=2)
    assert q["n_classes"] == 9 and q["launches"] == 1 + 3 * 2 * 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="passes fake pointers; host-side checks only")
def test_noalloc_limits_are_checked_before_the_device(L):
    # fake, 16-byte-aligned pointers: every case below must be rejected on the
    # host, before any device work (there is no device here)
    fake = 1 << 20
    norms = 1 << 21
    n = 1025  # more matrices than the fixed scratch has tickets for (1024)
    st = mu.muon_momentum_norm_noalloc([fake] * n, [fake] * n, [fake] * n, norms, shapes=[(64, 64)] * n,
                                       check=False)
    assert st == mu.MUON_ERR_SCRATCH_LIMIT
    # 17 matrices of 1024 x 16 tiles of 64 x 64 = 278528 tiles in one launch group (> 262144)
    st = mu.muon_momentum_norm_noalloc([fake] * 17, [fake] * 17, [fake] * 17, norms,
                                       shapes=[(65536, 1024)] * 17, check=False)
    assert st == mu.MUON_ERR_SCRATCH_LIMIT
    assert mu.muon_status_string(mu.MUON_ERR_SCRATCH_LIMIT).startswith("request exceeds")
    # argument errors
    assert mu.muon_momentum_norm_noalloc([fake], [fake], [fake], norms, shapes=[(64, 60)],
                                         check=False) == mu.MUON_ERR_UNSUPPORTED_SHAPE
    assert mu.muon_momentum_norm_noalloc([fake], [fake], [fake], norms, shapes=[(64, 64)], momentum_mode=3,
                                         check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_momentum_norm_noalloc([fake + 4], [fake], [fake], norms, shapes=[(64, 64)],
                                         check=False) == mu.MUON_ERR_MISALIGNED
    assert mu.muon_momentum_norm_noalloc([fake], [fake], [0], norms, shapes=[(64, 64)],
                                         check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_momentum_norm_noalloc([], [], [], norms, shapes=[], check=False) == mu.MUON_OK
    # within the limits the call reaches the device check (none here)
    assert mu.muon_momentum_norm_noalloc([fake], [fake], [fake], norms, shapes=[(64, 64)],
                                         check=False) == mu.MUON_ERR_UNSUPPORTED_DEVICE


@pytest.mark.skipif(torch.cuda.is_available(), reason="passes fake pointers; host-side checks only")
def test_adamw_arguments_are_checked_before_the_device(L):
    fake = 1 << 20
    args = mu.AdamWArgs([fake], [fake], [fake], [fake], numels=[64])
    assert mu.muon_adamw_step(args, step=0, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_adamw_step(args, beta1=1.5, check=False) == mu.MUON_ERR_INVALID_ARG
    bad = mu.AdamWArgs([fake + 8], [fake], [fake], [fake], numels=[64])
    assert mu.muon_adamw_step(bad, check=False) == mu.MUON_ERR_MISALIGNED
    neg = mu.AdamWArgs([fake], [fake], [fake], [fake], numels=[-1])
    assert mu.muon_adamw_step(neg, check=False) == mu.MUON_ERR_INVALID_ARG
    assert mu.muon_adamw_step([], [], [], [], check=False) == mu.MUON_OK
    # valid arguments reach the device check (no device here)
    assert mu.muon_adamw_step(args, check=False) == mu.MUON_ERR_UNSUPPORTED_DEVICE


def test_adamw_set_shapes():
    shapes = workloads.adamw_shapes("d26")
    assert shapes[0] == (32768, 1664) and shapes[1] == (32768, 1664)
    assert sum(math.prod(s) for s in shapes) == 2 * 32768 * 1664 + 52 + 24 + 1


def test_header_constants_match_the_binding():
    # every MUON_* value the header defines has the same value in the Python binding
    import re
    text = open(mu.HEADER_PATH).read()
    pairs = re.findall(r"\b(MUON_[A-Z0-9_]+)\s*=\s*(\d+)", text)
    assert len(pairs) >= 17
    for name, value in pairs:
        assert getattr(mu, name) == int(value), name


def test_struct_layouts_match_the_header():
    # the ctypes structures have the sizes and field offsets a C compiler gives the header's
    import shutil
    import subprocess
    import tempfile
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    structs = {"muon_shape": mu.muon_shape, "muon_config": mu.muon_config, "muon_step_info": mu.muon_step_info,
               "muon_plan_info": mu.muon_plan_info}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "muon.h"', "int main(void) {"]
    for sname, cls in structs.items():
        lines.append(f'printf("{sname} sizeof %zu\\n", sizeof({sname}));')
        for fname, _ in cls._fields_:
            lines.append(f'printf("{sname} {fname} %zu\\n", offsetof({sname}, {fname}));')
    lines += ["return 0;", "}"]
    build = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "_build", "tests")
    os.makedirs(build, exist_ok=True)
    with tempfile.TemporaryDirectory(dir=build) as tmp:
        src, exe = os.path.join(tmp, "layout.c"), os.path.join(tmp, "layout")
        open(src, "w").write("\n".join(lines) + "\n")
        subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(mu.HEADER_PATH), "-o", exe, src], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    seen = 0
    for ln in out.splitlines():
        sname, field, value = ln.split()
        cls = structs[sname]
        got = ctypes.sizeof(cls) if field == "sizeof" else getattr(cls, field).offset
        assert got == int(value), (sname, field, got, value)
        seen += 1
    assert seen == sum(len(c._fields_) + 1 for c in structs.values())
