"""Fused MoE finalize + rank sum + residual + RMSNorm (+ FP8 / NVFP4 quantisation) for GB300.

This package is a thin ctypes binding over the C ABI declared in ``include/moe_finalize.h`` and
implemented by ``libmoe_finalize.so`` (hand-written sm_103a CUDA kernels).  The binding only checks
and marshals arguments: every step of the computation runs in the library's kernels.  PyTorch is
used for device memory and the current stream.  There is no CPU fallback: if the library is missing
the import fails.

Per token t and hidden index h (flashinfer PR #6631 "perf(comm): gather MoE-finalize routes together
and accumulate in FP32", Description; TensorRT-LLM PR #16778, Fix):

    p_r = round(fma-chain_k(scale_r[t,k] * gemm2_r[perm_r[t,k], h]) * rsf + shared_r[t,h])
    S   = round(p_0 + ... + p_{R-1})                  (FP32, rank order)
    residual_out = round(S + residual)
    norm_out     = round((x * rstd) * gamma),  x = residual_out, rstd = 1/sqrt(mean(x^2) + eps)
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Sequence

import torch

__all__ = [
    "Partial", "moe_finalize_fused", "moe_finalize_routed", "moe_finalize_plan", "moe_finalize_sf_bytes", "moe_finalize_quant_bytes",
    "moe_finalize_empty_launch", "moe_finalize_gather_floor_launch", "moe_finalize_read_timeouts", "moe_finalize_abi_version", "library_path",
    "QUANT", "SF_LAYOUT", "KERNEL", "MFR_FLAG_PDL", "MFR_FLAG_ROUTING_READY", "MFR_FLAG_TEST_EXCHANGE_TIMEOUT",
    "MFR_FLAG_TEST_STREAM_TIMEOUT",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libmoe_finalize.so")

MFR_BF16, MFR_FP16, MFR_FP32 = 0, 1, 2
DTYPE = {torch.bfloat16: MFR_BF16, torch.float16: MFR_FP16, torch.float32: MFR_FP32}
QUANT = {"none": 0, "fp8": 1, "nvfp4": 2}
SF_LAYOUT = {"row_major": 0, "swizzled_128x4": 1}
KERNEL = {"auto": 0, "cluster": 1, "stream": 2, "bulk": 3}
MFR_FLAG_PDL, MFR_FLAG_ROUTING_READY = 1, 2
MFR_FLAG_TEST_EXCHANGE_TIMEOUT = 1 << 30  # test hook: every cluster exchange wait runs out (see the C header)
MFR_FLAG_TEST_STREAM_TIMEOUT = 1 << 29    # test hook: every stream end-of-token wait runs out (see the C header)
STATUS = {0: "MFR_OK", -1: "MFR_ERR_INVALID_ARG", -2: "MFR_ERR_UNSUPPORTED", -3: "MFR_ERR_CUDA"}


class _CPartial(ctypes.Structure):
    _fields_ = [("gemm2_out", ctypes.c_void_p), ("num_rows", ctypes.c_int64), ("perm_idx", ctypes.c_void_p),
                ("expert_scale", ctypes.c_void_p), ("shared_out", ctypes.c_void_p)]


class _CArgs(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("K", ctypes.c_int32), ("R", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("scale_dtype", ctypes.c_int32),
                ("routed_scaling_factor", ctypes.c_float), ("eps", ctypes.c_float),
                ("partials", ctypes.POINTER(_CPartial)),
                ("residual", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
                ("residual_out", ctypes.c_void_p), ("norm_out", ctypes.c_void_p),
                ("quant_mode", ctypes.c_int32), ("sf_layout", ctypes.c_int32),
                ("quant_scale", ctypes.c_void_p), ("quant_out", ctypes.c_void_p), ("sf_out", ctypes.c_void_p),
                ("flags", ctypes.c_uint32), ("kernel", ctypes.c_int32), ("finalize_out", ctypes.c_void_p)]


class _CPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("kernel", "grid", "cluster", "block", "smem_bytes", "chunk", "stages")]


def _load_library():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' or "
            f"python moe_finalize_residual_gb300/build.py).  There is no CPU fallback.")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    lib.moe_finalize_fused.argtypes = [ctypes.POINTER(_CArgs), P]
    lib.moe_finalize_fused.restype = ctypes.c_int
    lib.moe_finalize_plan.argtypes = [ctypes.POINTER(_CArgs), ctypes.POINTER(_CPlan)]
    lib.moe_finalize_plan.restype = ctypes.c_int
    lib.moe_finalize_sf_bytes.argtypes = [ctypes.c_int32] * 3
    lib.moe_finalize_sf_bytes.restype = ctypes.c_int64
    lib.moe_finalize_quant_bytes.argtypes = [ctypes.c_int32] * 3
    lib.moe_finalize_quant_bytes.restype = ctypes.c_int64
    lib.moe_finalize_status_string.argtypes = [ctypes.c_int]
    lib.moe_finalize_status_string.restype = ctypes.c_char_p
    lib.moe_finalize_last_error.argtypes = []
    lib.moe_finalize_last_error.restype = ctypes.c_char_p
    lib.moe_finalize_empty_launch.argtypes = [P, ctypes.c_uint32]
    lib.moe_finalize_empty_launch.restype = ctypes.c_int
    lib.moe_finalize_gather_floor_launch.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, P, P, ctypes.c_uint32]
    lib.moe_finalize_gather_floor_launch.restype = ctypes.c_int
    lib.moe_finalize_read_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.moe_finalize_read_timeouts.restype = ctypes.c_int
    lib.moe_finalize_abi_version.argtypes = []
    lib.moe_finalize_abi_version.restype = ctypes.c_int
    return lib


_lib = _load_library()


def library_path() -> str:
    return _LIB_PATH


class MoEFinalizeError(RuntimeError):
    pass


def _check(status: int):
    if status != 0:
        msg = _lib.moe_finalize_last_error().decode()
        raise MoEFinalizeError(f"{STATUS.get(status, status)}: {msg}")


@dataclasses.dataclass
class Partial:
    """One tensor-parallel partial (what one TP rank holds).  R = 1 is the plain MoE finalize."""

    gemm2_out: torch.Tensor                     # [num_rows, H] act, permuted GEMM2 output rows
    perm_idx: torch.Tensor                      # [T, K] int32; -1 (or out of range) = skipped route
    expert_scale: Optional[torch.Tensor] = None  # [T, K] fp32/bf16/fp16; None = all 1.0
    shared_out: Optional[torch.Tensor] = None    # [T, H] act; None = no shared expert


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _as_device_scale(q, device) -> torch.Tensor:
    """The quantisation scale may be a Python number or a 0-D / 1-element tensor (flashinfer PR #3385,
    review: accept scalar tensors, not only floats)."""
    if isinstance(q, torch.Tensor):
        if q.numel() != 1:
            raise ValueError("quant_scale must hold exactly one value")
        return q.reshape(1).to(device=device, dtype=torch.float32)
    return torch.tensor([float(q)], dtype=torch.float32, device=device)


def _build_args(partials: Sequence[Partial], residual, gamma, routed_scaling_factor, eps, residual_out, norm_out,
                quant_mode, quant_scale, sf_layout, quant_out, sf_out, flags, kernel, check=True, finalize_out=None):
    if len(partials) == 0:
        raise ValueError("at least one partial is required")
    p0 = partials[0]
    device = residual.device if residual is not None else p0.gemm2_out.device
    T = p0.perm_idx.shape[0] if p0.perm_idx.dim() == 2 else 0
    H = residual.shape[1] if residual is not None else p0.gemm2_out.shape[1]
    K = p0.perm_idx.shape[1] if p0.perm_idx.dim() == 2 else 0
    act = residual.dtype if residual is not None else p0.gemm2_out.dtype
    sdt = None
    if check:
        if residual is not None and residual.shape != (T, H):
            raise ValueError(f"residual must be [{T}, {H}] (T from perm_idx)")
        # flashinfer PR #3385, review: every caller-provided tensor must be on the input's device.
        tensors = [("residual", residual), ("gamma", gamma), ("residual_out", residual_out), ("norm_out", norm_out),
                   ("quant_out", quant_out), ("sf_out", sf_out), ("quant_scale", quant_scale),
                   ("finalize_out", finalize_out)]
        for r, p in enumerate(partials):
            tensors += [(f"partials[{r}].gemm2_out", p.gemm2_out), (f"partials[{r}].perm_idx", p.perm_idx),
                        (f"partials[{r}].expert_scale", p.expert_scale), (f"partials[{r}].shared_out", p.shared_out)]
        for name, t in tensors:
            if t is None:
                continue
            if t.device != device or device.type != "cuda":
                raise ValueError(f"{name} is on {t.device}; every tensor must be on {device} (a CUDA device)")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        if act not in (torch.bfloat16, torch.float16):
            raise ValueError(f"activation dtype {act} not supported (bfloat16 or float16)")
        if gamma is not None and (gamma.shape != (H,) or gamma.dtype != act):
            raise ValueError("gamma must be [H] of the activation dtype")
        for r, p in enumerate(partials):
            if p.gemm2_out.dim() != 2 or p.gemm2_out.shape[1] != H or p.gemm2_out.dtype != act:
                raise ValueError(f"partials[{r}].gemm2_out must be [rows, {H}] {act}")
            if p.perm_idx.shape != (T, K) or p.perm_idx.dtype != torch.int32:
                raise ValueError(f"partials[{r}].perm_idx must be [{T}, {K}] int32")
            if p.expert_scale is not None:
                if p.expert_scale.shape != (T, K) or p.expert_scale.dtype not in DTYPE:
                    raise ValueError(f"partials[{r}].expert_scale must be [{T}, {K}] fp32/bf16/fp16")
                if sdt is not None and p.expert_scale.dtype != sdt:
                    raise ValueError("all expert_scale tensors must share one dtype")
                sdt = p.expert_scale.dtype
            if p.shared_out is not None and (p.shared_out.shape != (T, H) or p.shared_out.dtype != act):
                raise ValueError(f"partials[{r}].shared_out must be [{T}, {H}] {act}")
        for name, t in (("residual_out", residual_out), ("norm_out", norm_out), ("finalize_out", finalize_out)):
            if t is not None and (t.shape != (T, H) or t.dtype != act):
                raise ValueError(f"{name} must be [{T}, {H}] {act}")
        # The library gets plain pointers, so the quantised buffers' sizes are checked here.
        qm = QUANT[quant_mode] if isinstance(quant_mode, str) else int(quant_mode)
        if qm != 0:
            need = {"quant_out": moe_finalize_quant_bytes(T, H, qm)}
            if qm == QUANT["nvfp4"]:
                need["sf_out"] = moe_finalize_sf_bytes(T, H, sf_layout)
            for name, t in (("quant_out", quant_out), ("sf_out", sf_out)):
                if name in need and t is not None and t.numel() * t.element_size() < need[name]:
                    raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes; {need[name]} are written")
    else:
        for p in partials:
            if p.expert_scale is not None:
                sdt = p.expert_scale.dtype
                break
    parts = (_CPartial * len(partials))()
    for r, p in enumerate(partials):
        parts[r] = _CPartial(p.gemm2_out.data_ptr(), p.gemm2_out.shape[0], p.perm_idx.data_ptr(),
                             _ptr(p.expert_scale), _ptr(p.shared_out))
    a = _CArgs()
    a.T, a.H, a.K, a.R = T, H, K, len(partials)
    a.act_dtype = DTYPE[act]
    a.scale_dtype = DTYPE[sdt] if sdt is not None else MFR_FP32
    a.routed_scaling_factor = float(routed_scaling_factor)
    a.eps = float(eps)
    a.partials = ctypes.cast(parts, ctypes.POINTER(_CPartial))
    a.residual, a.gamma = _ptr(residual), _ptr(gamma)
    a.finalize_out = _ptr(finalize_out)
    a.residual_out, a.norm_out = _ptr(residual_out), _ptr(norm_out)
    a.quant_mode = QUANT[quant_mode] if isinstance(quant_mode, str) else int(quant_mode)
    a.sf_layout = SF_LAYOUT[sf_layout] if isinstance(sf_layout, str) else int(sf_layout)
    a.quant_scale, a.quant_out, a.sf_out = _ptr(quant_scale), _ptr(quant_out), _ptr(sf_out)
    a.flags = int(flags)
    a.kernel = KERNEL[kernel] if isinstance(kernel, str) else int(kernel)
    return a, parts


def moe_finalize_fused(partials: Sequence[Partial], residual: torch.Tensor, gamma: torch.Tensor, *,
                       routed_scaling_factor: float = 1.0, eps: float = 1e-6,
                       residual_out: Optional[torch.Tensor] = None, norm_out: Optional[torch.Tensor] = None,
                       want_residual_out: bool = True, want_norm_out: bool = True,
                       quant_mode: str = "none", quant_scale=None, sf_layout: str = "row_major",
                       quant_out: Optional[torch.Tensor] = None, sf_out: Optional[torch.Tensor] = None,
                       pdl: bool = True, routing_ready: bool = False, kernel: str = "auto",
                       stream: Optional[torch.cuda.Stream] = None, check: bool = True,
                       finalize_out: Optional[torch.Tensor] = None, extra_flags: int = 0):
    """Enqueue the fused finalize on ``stream`` (default: the current stream).

    Outputs that are not passed in are allocated (``want_*`` = False leaves them out).  Returns
    ``(residual_out, norm_out, quant_out, sf_out)`` with None for outputs not produced.
    ``quant_scale`` is the FP8 encode scale or the NVFP4 global scale (a float or a 1-element tensor).
    ``finalize_out`` ([T, H] act), when given, also receives the finalized MoE output before the
    residual (the rounded rank sum).  ``extra_flags`` are further ``MFR_FLAG_*`` bits (the failure-detection
    test hook ``MFR_FLAG_TEST_EXCHANGE_TIMEOUT``).
    """
    T, H = residual.shape
    dev = residual.device
    if residual_out is None and want_residual_out:
        residual_out = torch.empty_like(residual)
    if norm_out is None and want_norm_out:
        norm_out = torch.empty_like(residual)
    qm = QUANT[quant_mode] if isinstance(quant_mode, str) else int(quant_mode)
    if qm != 0:
        if quant_scale is None:
            raise ValueError("quantisation needs quant_scale")
        if not (isinstance(quant_scale, torch.Tensor) and quant_scale.dtype == torch.float32
                and quant_scale.device == dev and quant_scale.numel() == 1):
            quant_scale = _as_device_scale(quant_scale, dev)
        if quant_out is None:
            quant_out = torch.empty(int(moe_finalize_quant_bytes(T, H, qm)), dtype=torch.uint8, device=dev)
        if qm == QUANT["nvfp4"] and sf_out is None:
            # zero-filled: the kernel writes no padding bytes of the 128x4 layout, and a block-scaled GEMM
            # reading the padded tile then sees zero scales, not stale memory
            sf_out = torch.zeros(int(moe_finalize_sf_bytes(T, H, sf_layout)), dtype=torch.uint8, device=dev)
    else:
        quant_scale = None
    flags = (MFR_FLAG_PDL if pdl else 0) | (MFR_FLAG_ROUTING_READY if routing_ready else 0) | int(extra_flags)
    a, keep = _build_args(partials, residual, gamma, routed_scaling_factor, eps, residual_out, norm_out, qm,
                          quant_scale, sf_layout, quant_out, sf_out, flags, kernel, check=check,
                          finalize_out=finalize_out)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    _check(_lib.moe_finalize_fused(ctypes.byref(a), ctypes.c_void_p(s.cuda_stream)))
    del keep
    return residual_out, norm_out, quant_out, sf_out


def moe_finalize_routed(partials: Sequence[Partial], *, routed_scaling_factor: float = 1.0,
                        out: Optional[torch.Tensor] = None, pdl: bool = True, routing_ready: bool = False,
                        kernel: str = "auto", stream: Optional[torch.cuda.Stream] = None,
                        check: bool = True) -> torch.Tensor:
    """Finalize-only mode: the finalized MoE output S = round(sum over r of p_r) ([T, H], the dtype of the
    GEMM2 rows; p_0 when there is one partial), with no residual add, RMSNorm or quantisation -- the
    standalone finalize that a deferred all-reduce or a separate residual-RMSNorm kernel consumes
    (flashinfer PR #6546, Description; TensorRT-LLM PR #16778, Fix).  Returns ``out``."""
    p0 = partials[0]
    T, H = p0.perm_idx.shape[0], p0.gemm2_out.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=p0.gemm2_out.dtype, device=p0.gemm2_out.device)
    flags = (MFR_FLAG_PDL if pdl else 0) | (MFR_FLAG_ROUTING_READY if routing_ready else 0)
    a, keep = _build_args(partials, None, None, routed_scaling_factor, 1e-6, None, None, 0, None, "row_major", None,
                          None, flags, kernel, check=check, finalize_out=out)
    s = stream if stream is not None else torch.cuda.current_stream(out.device)
    _check(_lib.moe_finalize_fused(ctypes.byref(a), ctypes.c_void_p(s.cuda_stream)))
    del keep
    return out


def moe_finalize_plan(partials: Sequence[Partial], residual: torch.Tensor, gamma: torch.Tensor, *,
                      quant_mode: str = "none", sf_layout: str = "row_major", kernel: str = "auto",
                      pdl: bool = True, with_norm_out: bool = True) -> dict:
    """The launch geometry the library would use for this problem on the current device."""
    dev = residual.device
    qm = QUANT[quant_mode] if isinstance(quant_mode, str) else int(quant_mode)
    dummy = residual  # only the pointers' presence and alignment matter for planning
    qs = torch.ones(1, dtype=torch.float32, device=dev) if qm else None
    a, keep = _build_args(partials, residual, gamma, 1.0, 1e-6, dummy, dummy if with_norm_out else None, qm, qs,
                          sf_layout, dummy if qm else None, dummy if qm == 2 else None,
                          MFR_FLAG_PDL if pdl else 0, kernel, check=False)
    plan = _CPlan()
    _check(_lib.moe_finalize_plan(ctypes.byref(a), ctypes.byref(plan)))
    del keep
    out = {n: getattr(plan, n) for n, _ in _CPlan._fields_}
    out["kernel"] = {1: "cluster", 2: "stream", 3: "bulk"}.get(out["kernel"], "none")
    return out


def moe_finalize_sf_bytes(T: int, H: int, sf_layout="row_major") -> int:
    lay = SF_LAYOUT[sf_layout] if isinstance(sf_layout, str) else int(sf_layout)
    n = _lib.moe_finalize_sf_bytes(T, H, lay)
    if n < 0:
        _check(int(n))
    return int(n)


def moe_finalize_quant_bytes(T: int, H: int, quant_mode="fp8") -> int:
    qm = QUANT[quant_mode] if isinstance(quant_mode, str) else int(quant_mode)
    n = _lib.moe_finalize_quant_bytes(T, H, qm)
    if n < 0:
        _check(int(n))
    return int(n)


def moe_finalize_empty_launch(stream: Optional[torch.cuda.Stream] = None, pdl: bool = True):
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(_lib.moe_finalize_empty_launch(ctypes.c_void_p(s.cuda_stream), MFR_FLAG_PDL if pdl else 0))


def moe_finalize_gather_floor_launch(idx: torch.Tensor, rows: torch.Tensor, out: torch.Tensor,
                                     stream: Optional[torch.cuda.Stream] = None, pdl: bool = True):
    """The index -> row -> store chain alone (a latency floor for the finalize); see the C header."""
    if idx.dtype != torch.int32 or not (idx.is_cuda and rows.is_cuda and out.is_cuda):
        raise MoEFinalizeError("idx must be a CUDA int32 tensor; rows and out CUDA tensors")
    if not rows.is_contiguous() or rows.dim() != 2 or out.numel() * out.element_size() < 512:
        raise MoEFinalizeError("rows must be a contiguous 2-D tensor and out at least 512 bytes")
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(_lib.moe_finalize_gather_floor_launch(
        ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(rows.data_ptr()), rows.shape[0],
        rows.shape[1] * rows.element_size(), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(s.cuda_stream),
        MFR_FLAG_PDL if pdl else 0))


def moe_finalize_read_timeouts() -> int:
    c = ctypes.c_uint32(0)
    _check(_lib.moe_finalize_read_timeouts(ctypes.byref(c)))
    return int(c.value)


def moe_finalize_abi_version() -> int:
    return int(_lib.moe_finalize_abi_version())


def raw_library():
    """The loaded ctypes library (for callers that build the C argument block themselves)."""
    return _lib
