"""CPU oracle for the fused MoE finalize + rank sum + residual + RMSNorm (+ FP8 / NVFP4 quant).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg are the only code that may import this package.  The CUDA library and its Python binding never
import it.  The arithmetic lives in ``mfr_oracle.c`` (plain C, FP32 in the order the definition gives,
compiled with ``-ffp-contract=off``); this module compiles it on demand with gcc and marshals
arguments through ctypes.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` (page-printed error
table, FP64 evaluation, dense brute force, invariants, closed forms, library conversions).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mfr_oracle.c")
_LIB = os.path.join(_HERE, "libmfr_oracle.so")
_lock = threading.Lock()
_lib = None

ACT = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
QUANT_NONE, QUANT_FP8, QUANT_NVFP4 = 0, 1, 2
SF_ROW_MAJOR, SF_SWIZZLED_128x4 = 0, 1
MODE_FP32_ACCUM, MODE_STEP_ROUNDED = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library beside its source (no fast-math, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Partial(ctypes.Structure):
    _fields_ = [("gemm2", ctypes.c_void_p), ("rows", ctypes.c_int64), ("perm", ctypes.c_void_p),
                ("scale", ctypes.c_void_p), ("shared", ctypes.c_void_p)]


class _Args(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("K", ctypes.c_int32), ("R", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("scale_dtype", ctypes.c_int32),
                ("rsf", ctypes.c_float), ("eps", ctypes.c_float),
                ("partials", ctypes.POINTER(_Partial)),
                ("residual", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
                ("t0", ctypes.c_int32), ("t1", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("residual_out", ctypes.c_void_p), ("norm_out", ctypes.c_void_p),
                ("routed_out", ctypes.c_void_p)]


def _load(path):
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(build())
        return _lib


class use_library:
    """Context manager: route every call of this module through another build of the oracle
    (the tests use it to run the pins against deliberately broken copies)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        lib()
        self.saved = _lib
        _lib = _load(self.path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved


def build_variant(src_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source with the same flags (used only by tests)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-o", out_path, src, "-lm"])
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _declare(L):
    P = ctypes.c_void_p
    L.oracle_finalize.argtypes = [ctypes.POINTER(_Args)]
    L.oracle_finalize_fp64.argtypes = [ctypes.POINTER(_Args), P, P]
    L.oracle_quantize.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_int32, P, P]
    L.oracle_sf_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    L.oracle_sf_bytes.restype = ctypes.c_int64
    L.oracle_sf_offset.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    L.oracle_sf_offset.restype = ctypes.c_int64
    for name in ("bf16", "fp16", "e4m3", "e2m1"):
        getattr(L, f"oracle_f32_to_{name}_array").argtypes = [P, P, ctypes.c_int64]
    L.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_to_f32.restype = ctypes.c_float
    L.oracle_e2m1_to_f32.argtypes = [ctypes.c_uint8]
    L.oracle_e2m1_to_f32.restype = ctypes.c_float
    L.oracle_sf_offsets.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P]
    L.oracle_fmaf.argtypes = [ctypes.c_float] * 3
    L.oracle_fmaf.restype = ctypes.c_float


def _ptr(t):
    return None if t is None else t.data_ptr()


def _args(case, t0, t1, mode, keep):
    """Build the ctypes argument block; ``keep`` holds references so CPU tensors outlive the call."""
    R = case.R
    parts = (_Partial * R)()
    for r in range(R):
        tensors = [x.cpu().contiguous() if x is not None else None
                   for x in (case.gemm2[r], case.perm[r], case.scale[r], case.shared[r])]
        keep.extend(tensors)
        g, p, s, sh = tensors
        parts[r] = _Partial(g.data_ptr(), g.shape[0], p.data_ptr(), _ptr(s), _ptr(sh))
    res = case.residual.cpu().contiguous()
    gam = case.gamma.cpu().contiguous()
    keep.extend([res, gam, parts])
    a = _Args()
    a.T, a.H, a.K, a.R = case.T, case.H, case.K, R
    a.act_dtype = ACT[case.act_dtype]
    a.scale_dtype = ACT[case.scale_dtype] if case.scale_dtype is not None else 2
    a.rsf, a.eps = case.rsf, case.eps
    a.partials = ctypes.cast(parts, ctypes.POINTER(_Partial))
    a.residual, a.gamma = res.data_ptr(), gam.data_ptr()
    a.t0, a.t1, a.mode = t0, t1, mode
    return a


def finalize(case, t0: int = 0, t1: int | None = None, mode: int = MODE_FP32_ACCUM):
    """Run the definition on tokens [t0, t1).  Returns uint16 bit arrays [T, H] (rows outside the
    range are zero): residual_out, norm_out and routed (the rounded rank sum before the residual)."""
    t1 = case.T if t1 is None else t1
    keep = []
    a = _args(case, t0, t1, mode, keep)
    out = {k: np.zeros((case.T, case.H), dtype=np.uint16) for k in ("residual_out", "norm_out", "routed")}
    a.residual_out = out["residual_out"].ctypes.data
    a.norm_out = out["norm_out"].ctypes.data
    a.routed_out = out["routed"].ctypes.data
    lib().oracle_finalize(ctypes.byref(a))
    return out


def finalize_threads(case, threads: int, t0: int = 0, t1: int | None = None, mode: int = MODE_FP32_ACCUM):
    """``finalize`` with tokens [t0, t1) split into ``threads`` contiguous ranges, each run by its own host
    thread (ctypes releases the GIL during the C call).  Tokens are independent and each is computed by
    the same code in the same order, so the result is bit-identical to ``finalize``."""
    t1 = case.T if t1 is None else t1
    out = {k: np.zeros((case.T, case.H), dtype=np.uint16) for k in ("residual_out", "norm_out", "routed")}
    n = max(1, min(int(threads), t1 - t0))
    bounds = [t0 + (t1 - t0) * i // n for i in range(n + 1)]
    keep, blocks = [], []
    for i in range(n):
        a = _args(case, bounds[i], bounds[i + 1], mode, keep)
        a.residual_out = out["residual_out"].ctypes.data
        a.norm_out = out["norm_out"].ctypes.data
        a.routed_out = out["routed"].ctypes.data
        blocks.append(a)
    L = lib()
    workers = [threading.Thread(target=L.oracle_finalize, args=(ctypes.byref(a),)) for a in blocks[1:]]
    for w in workers:
        w.start()
    L.oracle_finalize(ctypes.byref(blocks[0]))
    for w in workers:
        w.join()
    return out


def finalize_fp64(case, t0: int = 0, t1: int | None = None):
    """FP64 evaluation of the same formula without intermediate rounding: (residual_ref, norm_ref)."""
    t1 = case.T if t1 is None else t1
    keep = []
    a = _args(case, t0, t1, MODE_FP32_ACCUM, keep)
    res = np.zeros((case.T, case.H), dtype=np.float64)
    nrm = np.zeros((case.T, case.H), dtype=np.float64)
    lib().oracle_finalize_fp64(ctypes.byref(a), res.ctypes.data, nrm.ctypes.data)
    return res, nrm


def sf_bytes(T: int, H: int, layout: int) -> int:
    return int(lib().oracle_sf_bytes(T, H, layout))


def sf_offset(m: int, k: int, H: int, layout: int) -> int:
    return int(lib().oracle_sf_offset(m, k, H, layout))


def sf_offsets(T: int, H: int, layout: int) -> np.ndarray:
    """[T, H/16] array of block-scale byte offsets."""
    out = np.zeros((T, H // 16), dtype=np.int64)
    lib().oracle_sf_offsets(T, H, layout, out.ctypes.data)
    return out


def quantize(norm_bits: np.ndarray, act_dtype, quant: int, qscale: float, sf_layout: int = SF_ROW_MAJOR,
             t0: int = 0, t1: int | None = None):
    """Quantise an act-typed [T, H] array given as uint16 bits.  Returns (quant bytes, sf bytes or None)."""
    norm_bits = np.ascontiguousarray(norm_bits, dtype=np.uint16)
    T, H = norm_bits.shape
    t1 = T if t1 is None else t1
    if quant == QUANT_FP8:
        q = np.zeros((T, H), dtype=np.uint8)
        sf = None
    else:
        q = np.zeros((T, H // 2), dtype=np.uint8)
        sf = np.zeros(sf_bytes(T, H, sf_layout), dtype=np.uint8)
    lib().oracle_quantize(norm_bits.ctypes.data, ACT[act_dtype], T, H, t0, t1, quant, float(qscale), sf_layout,
                          q.ctypes.data, None if sf is None else sf.ctypes.data)
    return q, sf


def _conv(name, x, out_dtype):
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=out_dtype)
    getattr(lib(), f"oracle_f32_to_{name}_array")(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f32_to_bf16(x): return _conv("bf16", x, np.uint16)
def f32_to_fp16(x): return _conv("fp16", x, np.uint16)
def f32_to_e4m3(x): return _conv("e4m3", x, np.uint8)
def f32_to_e2m1(x): return _conv("e2m1", x, np.uint8)
def e4m3_to_f32(c: int) -> float: return float(lib().oracle_e4m3_to_f32(c))
def e2m1_to_f32(c: int) -> float: return float(lib().oracle_e2m1_to_f32(c))
def fmaf(a, b, c) -> float: return float(lib().oracle_fmaf(a, b, c))
