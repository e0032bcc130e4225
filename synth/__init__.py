"""Seeded synthetic inputs for the fused MoE finalize + residual + RMSNorm path.

This module only *draws* inputs: routing logits, expert choices, permutations,
GEMM2 rows, residuals, norm weights.  It holds none of the finalize arithmetic
(no weighted sums, no rank sum, no normalisation, no quantisation), so both the
CPU oracle and the CUDA path can consume its output without sharing any of the
method with each other.

Workload recipes (all values seeded, nothing read from disk):

* ``make_case`` -- the routed-MoE decode workloads.  Per partial ``r`` (one
  tensor-parallel rank's contribution): logits ``[T, E] ~ N(0, 1)``, softmax,
  top-k, renormalised to sum 1, cast to the scale dtype.  The expanded route
  ``j = t*K + k`` is stable-sorted by expert id; its position in that order is
  the permuted GEMM2 row, so ``perm[t, k]`` is that position and the GEMM2
  output is ``[T*K, H]`` in expert-sorted order, values ``N(0, 0.05^2)``.
  Optionally a quarter of the routes is masked to -1 and the rows they would
  have read are poisoned with NaN.  residual ``~ N(0, 1)``, gamma
  ``1 + N(0, 0.1^2)``.
* ``make_p1_case`` -- the distribution of the benchmark script in flashinfer PR
  #6631 "gather MoE-finalize routes together and accumulate in FP32"
  (fi_finalize_bench.py): ``2*T*K + 8`` GEMM2 rows of ``0.5 N(0,1)``, a random
  choice of ``T*K`` distinct rows, softmax(N(0,1)) weights over the K routes,
  shared output ``0.5 N(0,1)``, residual ``4 N(0,1)``, gamma ``1 + 0.1 N(0,1)``,
  routed_scaling_factor 2.5, eps 1e-5.

Seeds follow that script: partial ``r`` of a T-token case draws from seed
``base + 1000*r + T``; residual and gamma from ``base + 7 + T`` (shared by all
partials).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import torch

__all__ = ["Case", "make_case", "make_p1_case", "config_cases", "CONFIGS"]


@dataclasses.dataclass
class Case:
    """One finalize problem.  Tensors live on ``device``; lists have one entry per partial."""

    name: str
    T: int
    H: int
    K: int
    R: int
    E: int
    act_dtype: torch.dtype
    scale_dtype: Optional[torch.dtype]
    rsf: float
    eps: float
    gemm2: List[torch.Tensor]            # [rows_r, H] act
    perm: List[torch.Tensor]             # [T, K] int32, -1 = masked
    scale: List[Optional[torch.Tensor]]  # [T, K] scale_dtype or None
    shared: List[Optional[torch.Tensor]] # [T, H] act or None
    expert: List[torch.Tensor]           # [T, K] int64 expert id of each route (before masking)
    residual: torch.Tensor               # [T, H] act
    gamma: torch.Tensor                  # [H] act

    @property
    def device(self) -> torch.device:
        return self.residual.device

    def to(self, device) -> "Case":
        mv = lambda x: None if x is None else x.to(device)
        return dataclasses.replace(
            self,
            gemm2=[mv(x) for x in self.gemm2], perm=[mv(x) for x in self.perm],
            scale=[mv(x) for x in self.scale], shared=[mv(x) for x in self.shared],
            expert=[mv(x) for x in self.expert], residual=mv(self.residual), gamma=mv(self.gamma))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _routing(T: int, E: int, K: int, g: torch.Generator, device):
    """Softmax top-k routing with renormalised weights (fp32) and expert ids."""
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    probs = torch.softmax(logits, dim=-1)
    w, ids = torch.topk(probs, K, dim=-1)
    w = w / w.sum(dim=-1, keepdim=True)
    return w, ids


def _expert_sorted_perm(ids: torch.Tensor) -> torch.Tensor:
    """perm[t, k] = position of expanded route t*K+k when routes are stably sorted by expert id."""
    T, K = ids.shape
    flat = ids.reshape(-1)
    order = torch.sort(flat, stable=True).indices          # order[pos] = expanded index
    pos = torch.empty_like(order)
    pos[order] = torch.arange(order.numel(), device=ids.device)
    return pos.view(T, K).to(torch.int32)


def make_case(name: str, T: int, H: int, K: int, R: int, E: int,
              act_dtype=torch.bfloat16, scale_dtype=torch.bfloat16,
              rsf: float = 1.0, shared: bool = False, mask_quarter: bool = False,
              eps: float = 1e-6, seed_base: int = 0, device="cpu",
              gemm2_std: float = 0.05, shared_std: float = 0.05) -> Case:
    """Routed-MoE decode workload (expert-sorted GEMM2 rows, softmax top-k weights)."""
    gemm2, perm, scale, shd, expert = [], [], [], [], []
    for r in range(R):
        g = _gen(seed_base + 1000 * r + T, device)
        w, ids = _routing(T, E, K, g, device)
        p = _expert_sorted_perm(ids)
        rows = torch.randn(T * K, H, generator=g, device=device, dtype=torch.float32) * gemm2_std
        rows = rows.to(act_dtype)
        if mask_quarter and T * K >= 4:
            n_mask = (T * K) // 4
            sel = torch.randperm(T * K, generator=g, device=device)[:n_mask]
            flat = p.view(-1).clone()
            poisoned = flat[sel].long()
            flat[sel] = -1
            p = flat.view(T, K)
            rows[poisoned] = float("nan")
        sh = None
        if shared:
            sh = (torch.randn(T, H, generator=g, device=device, dtype=torch.float32) * shared_std).to(act_dtype)
        gemm2.append(rows)
        perm.append(p.contiguous())
        scale.append(None if scale_dtype is None else w.to(scale_dtype).contiguous())
        shd.append(sh)
        expert.append(ids)
    gs = _gen(seed_base + 7 + T, device)
    residual = torch.randn(T, H, generator=gs, device=device, dtype=torch.float32).to(act_dtype)
    gamma = (1.0 + 0.1 * torch.randn(H, generator=gs, device=device, dtype=torch.float32)).to(act_dtype)
    return Case(name, T, H, K, R, E, act_dtype, scale_dtype, float(rsf), float(eps),
                gemm2, perm, scale, shd, expert, residual, gamma)


def make_p1_case(T: int, H: int, R: int = 4, K: int = 8, device="cpu", seed_base: int = 0) -> Case:
    """The benchmark distribution of flashinfer PR #6631 (fi_finalize_bench.py), one partial per TP rank."""
    gemm2, perm, scale, shd, expert = [], [], [], [], []
    for r in range(R):
        g = _gen(seed_base + 1000 * r + T, device)
        rows = 2 * T * K + 8
        x = (torch.randn(rows, H, generator=g, device=device) * 0.5).to(torch.bfloat16)
        idx = torch.randperm(rows, generator=g, device=device)[: T * K].view(T, K).to(torch.int32)
        w = torch.softmax(torch.randn(T, K, generator=g, device=device), dim=-1).to(torch.bfloat16)
        sh = (torch.randn(T, H, generator=g, device=device) * 0.5).to(torch.bfloat16)
        gemm2.append(x)
        perm.append(idx.contiguous())
        scale.append(w.contiguous())
        shd.append(sh)
        expert.append(torch.arange(T * K, device=device).view(T, K))  # each route its own "expert"
    gs = _gen(seed_base + 7 + T, device)
    residual = (torch.randn(T, H, generator=gs, device=device) * 4).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(H, generator=gs, device=device)).to(torch.bfloat16)
    return Case("p1", T, H, K, R, T * K, torch.bfloat16, torch.bfloat16, 2.5, 1e-5,
                gemm2, perm, scale, shd, expert, residual, gamma)


# The five workload families (seed bases keep their random streams apart).
CONFIGS = {
    "tiny": dict(H=256, K=2, R=1, E=8, rsf=1.0, shared=False, act_dtype=torch.bfloat16,
                 scale_dtype=torch.bfloat16, seed_base=0, Ts=(4,)),
    "decode": dict(H=6144, K=8, R=4, E=256, rsf=2.5, shared=True, act_dtype=torch.bfloat16,
                   scale_dtype=torch.bfloat16, seed_base=100_000, Ts=(1, 4, 16, 32, 64, 128)),
    "masked": dict(H=7168, E=256, rsf=1.0, shared=False, mask_quarter=True, seed_base=200_000,
                   Ts=(1, 16, 64, 128)),  # K, R, act, scale dtype vary
    "highk": dict(R=1, rsf=1.0, shared=False, act_dtype=torch.bfloat16, scale_dtype=torch.float32,
                  seed_base=300_000, Ts=(1, 8, 16, 32, 64, 128)),  # (H, E, K) vary
    "bandwidth": dict(K=8, R=4, E=256, rsf=1.0, shared=False, act_dtype=torch.bfloat16,
                      scale_dtype=torch.bfloat16, seed_base=400_000, Ts=(1024, 4096, 16384)),
}
HIGHK_SHAPES = ((2048, 512, 22), (3584, 896, 16), (4096, 512, 32))


def config_cases(family: str, device="cpu", Ts=None):
    """Yield every case of one workload family (all its shape and dtype variants)."""
    c = dict(CONFIGS[family])
    Ts = Ts or c.pop("Ts")
    c.pop("Ts", None)
    if family == "masked":
        for K in (6, 8, 10):
            for act in (torch.float16, torch.bfloat16):
                for R in (2, 4):
                    for sdt in (torch.float32, torch.bfloat16):
                        for T in Ts:
                            yield make_case(f"masked-K{K}-{str(act)[6:]}-R{R}-{str(sdt)[6:]}-T{T}",
                                            T=T, K=K, R=R, act_dtype=act, scale_dtype=sdt,
                                            device=device, **c)
    elif family == "highk":
        for (H, E, K) in HIGHK_SHAPES:
            for T in Ts:
                yield make_case(f"highk-H{H}-K{K}-T{T}", T=T, H=H, E=E, K=K, device=device, **c)
    elif family == "bandwidth":
        for H in (6144, 7168):
            for T in Ts:
                yield make_case(f"bandwidth-H{H}-T{T}", T=T, H=H, device=device, **c)
    else:
        for T in Ts:
            yield make_case(f"{family}-T{T}", T=T, device=device, **c)
