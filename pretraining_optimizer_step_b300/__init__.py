"""Python binding of libmuon.so, the B300 Muon optimizer-step library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/muon.h.  The functions keep the
C names.  Device memory and streams come from PyTorch tensors (anything with
``data_ptr()``/``shape``) or raw integers.

If the shared library is missing the import still succeeds, but every call
raises ``MuonLibraryMissing``; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmuon.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "muon.h")

# muon_status codes (include/muon.h)
MUON_OK = 0
MUON_ERR_INVALID_ARG = 1
MUON_ERR_UNSUPPORTED_SHAPE = 2
MUON_ERR_MISALIGNED = 3
MUON_ERR_NOT_INITIALIZED = 4
MUON_ERR_CUDA = 5
MUON_ERR_OUT_OF_MEMORY = 6
MUON_ERR_DEVICE_TIMEOUT = 7
MUON_ERR_DEVICE_BOUNDS = 8
MUON_ERR_UNSUPPORTED_DEVICE = 9
MUON_ERR_SCRATCH_LIMIT = 10

MUON_MOMENTUM_SGD_NESTEROV = 0
MUON_MOMENTUM_EMA = 1

MUON_DEBUG_KEEP_O = 1
MUON_DEBUG_POISON_WORKSPACE = 2
MUON_DEBUG_TIME_KERNELS = 4
MUON_DEBUG_INJECT_LOST_LOAD = 8
MUON_DEBUG_INJECT_BAD_TILES = 16

# The five per-iteration "Polar Express" (a, b, c) rows, for muon_init(coeffs=...).  The pages
# print the first two to three decimals (apidog.com "Cara Melatih ChatGPT Sendiri dengan Budget 50
# Dolar", section "2. Pengoptimal Muon", coefficient list) and elide the rest; these full-precision
# rows come from the Polar Express construction (greedy minimax odd quintics on the interval where
# the singular values lie: start 1e-3, cushion u/50, recentring on 1, safety factor 1.02 on every
# row but the last), and agree with the printed figures to their last decimal.  The default table
# stays the fixed quintic (3.4445, -4.7750, 2.0315) x 5.
POLAR_EXPRESS_COEFFS = (
    (8.156554524902461, -22.483292925577953, 15.878769915207466),
    (4.042929935166726, -2.8089174659087055, 0.50001784510513),
    (3.891667802292667, -2.772484153217687, 0.5060648178503395),
    (3.2857536577556523, -2.3681294933425345, 0.4644902423300303),
    (2.3465413258596395, -1.7097828382687077, 0.4232355116930525),
)

KERNEL_KINDS = ("momentum_norm", "gram", "poly", "axpy", "axpy_update", "update", "axpy_o", "normuon")


class MuonLibraryMissing(RuntimeError):
    pass


class MuonError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {muon_status_string(status)} (status {status})")


class muon_shape(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int), ("cols", ctypes.c_int)]


class muon_config(ctypes.Structure):
    _fields_ = [("coeffs", ctypes.POINTER(ctypes.c_double)), ("n_coeff_rows", ctypes.c_int),
                ("eps", ctypes.c_double), ("momentum_mode", ctypes.c_int),
                ("debug_flags", ctypes.c_int), ("wait_timeout_s", ctypes.c_double)]


class muon_step_info(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int), ("n_classes", ctypes.c_int),
                ("workspace_bytes", ctypes.c_longlong), ("ns_alg_flops", ctypes.c_double),
                ("elementwise_alg_bytes", ctypes.c_double)]


class muon_plan_info(ctypes.Structure):
    _fields_ = [("n_classes", ctypes.c_int), ("launches", ctypes.c_int),
                ("workspace_bytes", ctypes.c_longlong), ("ns_alg_flops", ctypes.c_double),
                ("ns_executed_flops", ctypes.c_double), ("elementwise_alg_bytes", ctypes.c_double),
                ("momentum_ctas", ctypes.c_int), ("sym_tiles", ctypes.c_longlong),
                ("axpy_tiles", ctypes.c_longlong)]


_lib = None


def lib():
    """The loaded libmuon.so (raises MuonLibraryMissing if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MuonLibraryMissing(
                f"{LIB_PATH} is missing; build it with `python -m pretraining_optimizer_step_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp = ctypes.c_void_p
        L.muon_init.argtypes = [ctypes.POINTER(muon_config)]
        L.muon_step.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                ctypes.POINTER(muon_shape), ctypes.c_int, ctypes.c_float,
                                ctypes.c_float, ctypes.c_int, ctypes.c_int, vp]
        L.muon_destroy.argtypes = []
        L.muon_get_status.argtypes = [vp]
        L.muon_status_string.argtypes = [ctypes.c_int]
        L.muon_status_string.restype = ctypes.c_char_p
        L.muon_get_step_info.argtypes = [ctypes.POINTER(muon_step_info)]
        L.muon_kernel_times.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int),
                                        ctypes.c_int]
        L.muon_debug_copy_ns_output.argtypes = [ctypes.c_int, vp, vp]
        L.muon_debug_copy_norms.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int]
        L.muon_plan_query.argtypes = [ctypes.POINTER(muon_shape), ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(muon_plan_info)]
        L.muon_momentum_norm_noalloc.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                                 vp, ctypes.POINTER(muon_shape), ctypes.c_int, ctypes.c_float,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_double, vp]
        L.muon_step_normuon.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                        ctypes.POINTER(vp), ctypes.POINTER(muon_shape), ctypes.c_int,
                                        ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_float, ctypes.c_float, vp]
        L.muon_partition.argtypes = [ctypes.POINTER(muon_shape), ctypes.c_int, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_int)]
        L.muon_adamw_step.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                      ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_longlong), ctypes.c_int,
                                      ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_float, ctypes.c_int, vp]
        for name in ("muon_init", "muon_step", "muon_destroy", "muon_get_status", "muon_get_step_info",
                     "muon_kernel_times", "muon_debug_copy_ns_output", "muon_debug_copy_norms",
                     "muon_plan_query", "muon_momentum_norm_noalloc", "muon_adamw_step", "muon_step_normuon", "muon_partition"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, where: str) -> int:
    if status != MUON_OK:
        raise MuonError(status, where)
    return status


def _ptr(x) -> int:
    return int(x.data_ptr()) if hasattr(x, "data_ptr") else int(x)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return None
    if hasattr(stream, "cuda_stream"):
        return int(stream.cuda_stream)
    return int(stream)


def muon_status_string(status: int) -> str:
    return lib().muon_status_string(int(status)).decode()


def muon_init(coeffs: Optional[Sequence[Sequence[float]]] = None, eps: float = 0.0,
              momentum_mode: int = MUON_MOMENTUM_SGD_NESTEROV, debug_flags: int = 0,
              wait_timeout_s: float = 0.0, check: bool = True) -> int:
    cfg = muon_config()
    keep = None
    if coeffs is not None:
        flat = [float(v) for row in coeffs for v in row]
        keep = (ctypes.c_double * len(flat))(*flat)
        cfg.coeffs = ctypes.cast(keep, ctypes.POINTER(ctypes.c_double))
        cfg.n_coeff_rows = len(flat) // 3
    cfg.eps = float(eps)
    cfg.momentum_mode = int(momentum_mode)
    cfg.debug_flags = int(debug_flags)
    cfg.wait_timeout_s = float(wait_timeout_s)
    st = lib().muon_init(ctypes.byref(cfg))
    return _check(st, "muon_init") if check else st


def muon_destroy() -> int:
    return _check(lib().muon_destroy(), "muon_destroy")


class StepArgs:
    """Pre-marshalled pointer and shape arrays for repeated muon_step calls."""

    def __init__(self, params: Sequence, grads: Sequence, momentum_bufs: Sequence,
                 shapes: Optional[Iterable] = None):
        n = len(params)
        if len(grads) != n or len(momentum_bufs) != n:
            raise ValueError("params, grads and momentum_bufs must have the same length")
        if shapes is None:
            shapes = [tuple(p.shape) for p in params]
        shapes = list(shapes)
        self.n = n
        self.params = (ctypes.c_void_p * max(n, 1))(*[_ptr(x) for x in params])
        self.grads = (ctypes.c_void_p * max(n, 1))(*[_ptr(x) for x in grads])
        self.moms = (ctypes.c_void_p * max(n, 1))(*[_ptr(x) for x in momentum_bufs])
        self.shapes = (muon_shape * max(n, 1))(*[muon_shape(int(r), int(c)) for r, c in shapes])


def muon_step(params, grads=None, momentum_bufs=None, lr: float = 0.02, beta: float = 0.95,
              nesterov: bool = True, ns_steps: int = 5, stream=None, shapes=None,
              check: bool = True) -> int:
    """Enqueue one Muon step.  ``params`` may be a prepared StepArgs."""
    args = params if isinstance(params, StepArgs) else StepArgs(params, grads, momentum_bufs, shapes)
    st = lib().muon_step(args.params, args.grads, args.moms, args.shapes, args.n, float(lr),
                         float(beta), 1 if nesterov else 0, int(ns_steps), _stream(stream))
    return _check(st, "muon_step") if check else st


def muon_step_normuon(params, grads=None, momentum_bufs=None, second_moments=None, lr: float = 0.02,
                      beta: float = 0.95, nesterov: bool = True, ns_steps: int = 5, beta2: float = 0.95,
                      eps2: float = 1e-10, stream=None, shapes=None, check: bool = True) -> int:
    """Enqueue one Muon step with NorMuon scaling (see include/muon.h).  ``params`` may be a
    prepared StepArgs, then ``second_moments`` is the list of per-row state arrays."""
    args = params if isinstance(params, StepArgs) else StepArgs(params, grads, momentum_bufs, shapes)
    vp = ctypes.c_void_p
    sm = (vp * max(args.n, 1))(*[_ptr(x) for x in second_moments])
    st = lib().muon_step_normuon(args.params, args.grads, args.moms, sm, args.shapes, args.n, float(lr),
                                 float(beta), 1 if nesterov else 0, int(ns_steps), float(beta2), float(eps2),
                                 _stream(stream))
    return _check(st, "muon_step_normuon") if check else st


def muon_get_status(stream=None, check: bool = True) -> int:
    st = lib().muon_get_status(_stream(stream))
    return _check(st, "muon_get_status") if check else st


def muon_get_step_info() -> dict:
    info = muon_step_info()
    _check(lib().muon_get_step_info(ctypes.byref(info)), "muon_get_step_info")
    return {f: getattr(info, f) for f, _ in muon_step_info._fields_}


def muon_plan_query(shapes, ns_steps: int = 5, check: bool = True):
    """Host-only description of the step muon_step would run for these stored shapes."""
    shapes = [(int(r), int(c)) for r, c in shapes]
    arr = (muon_shape * max(len(shapes), 1))(*[muon_shape(r, c) for r, c in shapes])
    info = muon_plan_info()
    st = lib().muon_plan_query(arr, len(shapes), int(ns_steps), ctypes.byref(info))
    if check:
        _check(st, "muon_plan_query")
        return {f: getattr(info, f) for f, _ in muon_plan_info._fields_}
    return st


def muon_partition(shapes, world: int) -> list:
    """Owner rank of every matrix for a sharded step over `world` ranks (host only)."""
    shapes = [(int(r), int(c)) for r, c in shapes]
    n = len(shapes)
    arr = (muon_shape * max(n, 1))(*[muon_shape(r, c) for r, c in shapes])
    out = (ctypes.c_int * max(n, 1))()
    _check(lib().muon_partition(arr, n, int(world), out), "muon_partition")
    return [out[i] for i in range(n)]


def muon_kernel_times() -> dict:
    """{kind: (milliseconds, launches)} since the previous call (needs MUON_DEBUG_TIME_KERNELS)."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    _check(lib().muon_kernel_times(ms, cnt, n), "muon_kernel_times")
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def muon_debug_copy_ns_output(mat: int, dst, stream=None) -> int:
    return _check(lib().muon_debug_copy_ns_output(int(mat), _ptr(dst), _stream(stream)),
                  "muon_debug_copy_ns_output")


def muon_debug_copy_norms(n: int):
    buf = (ctypes.c_float * max(n, 1))()
    _check(lib().muon_debug_copy_norms(buf, int(n)), "muon_debug_copy_norms")
    return [buf[i] for i in range(n)]


class AdamWArgs:
    """Pre-marshalled pointer and size arrays for repeated muon_adamw_step calls."""

    def __init__(self, params: Sequence, grads: Sequence, exp_avg: Sequence, exp_avg_sq: Sequence,
                 numels: Optional[Sequence[int]] = None):
        n = len(params)
        if not (len(grads) == len(exp_avg) == len(exp_avg_sq) == n):
            raise ValueError("params, grads, exp_avg and exp_avg_sq must have the same length")
        if numels is None:
            numels = [int(x.numel()) for x in params]
        vp = ctypes.c_void_p
        self.n = n
        self.params = (vp * max(n, 1))(*[_ptr(x) for x in params])
        self.grads = (vp * max(n, 1))(*[_ptr(x) for x in grads])
        self.exp_avg = (vp * max(n, 1))(*[_ptr(x) for x in exp_avg])
        self.exp_avg_sq = (vp * max(n, 1))(*[_ptr(x) for x in exp_avg_sq])
        self.numels = (ctypes.c_longlong * max(n, 1))(*[int(k) for k in numels])


def muon_adamw_step(params, grads=None, exp_avg=None, exp_avg_sq=None, lr: float = 1e-3,
                    beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8, weight_decay: float = 0.01,
                    step: int = 1, stream=None, numels=None, check: bool = True) -> int:
    """Enqueue one AdamW step over a list of fp32 tensors (see include/muon.h).
    ``params`` may be a prepared AdamWArgs."""
    a = params if isinstance(params, AdamWArgs) else AdamWArgs(params, grads, exp_avg, exp_avg_sq, numels)
    st = lib().muon_adamw_step(a.params, a.grads, a.exp_avg, a.exp_avg_sq, a.numels, a.n, float(lr),
                               float(beta1), float(beta2), float(eps), float(weight_decay), int(step),
                               _stream(stream))
    return _check(st, "muon_adamw_step") if check else st


def muon_momentum_norm_noalloc(grads, momentum_bufs, x0_out, norms_out, beta: float = 0.95,
                               nesterov: bool = True, momentum_mode: int = MUON_MOMENTUM_SGD_NESTEROV,
                               eps: float = 0.0, stream=None, shapes=None, check: bool = True) -> int:
    """The momentum + norm pass with no allocation (see include/muon.h).

    For callers that may not allocate device memory: momentum_bufs are updated
    in place, x0_out[i] (bf16 buffers of rows * cols elements) receive the
    unscaled direction in the oriented layout, norms_out (float32, n) its
    Frobenius norm.  Scratch lives in a fixed array inside the library."""
    n = len(grads)
    if len(momentum_bufs) != n or len(x0_out) != n:
        raise ValueError("grads, momentum_bufs and x0_out must have the same length")
    if shapes is None:
        shapes = [tuple(g.shape) for g in grads]
    vp = ctypes.c_void_p
    g_arr = (vp * max(n, 1))(*[_ptr(x) for x in grads])
    m_arr = (vp * max(n, 1))(*[_ptr(x) for x in momentum_bufs])
    x_arr = (vp * max(n, 1))(*[_ptr(x) for x in x0_out])
    s_arr = (muon_shape * max(n, 1))(*[muon_shape(int(r), int(c)) for r, c in shapes])
    st = lib().muon_momentum_norm_noalloc(g_arr, m_arr, x_arr, _ptr(norms_out) if norms_out is not None else None,
                                          s_arr, n, float(beta), 1 if nesterov else 0, int(momentum_mode),
                                          float(eps), _stream(stream))
    return _check(st, "muon_momentum_norm_noalloc") if check else st


def declared_symbols() -> list:
    """Function names declared in include/muon.h (used by the export test)."""
    import re
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:MUON_API\s+)?(?:const\s+char\*|muon_status)\s+(muon_\w+)\s*\(", text, re.M)))


from . import zero2  # noqa: E402  (the sharded step driver uses the functions above)
