"""Helpers shared by the GPU parity tests: running the library on a synth.Case, canary-guarded
outputs, sampled sub-problems for full-size cases, and the comparisons against the oracle."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
import synth

CANARY = 0x5A
GUARD = 4096  # bytes of canary before and after every output buffer


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def as_f64(b: np.ndarray, act) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(act).double().numpy()


def ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray, act=torch.bfloat16) -> np.ndarray:
    """Ordinal distance between 16-bit float bit patterns; +0 and -0 are equal; NaN vs NaN is 0."""
    def ordinal(b):
        b = b.astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    d = np.abs(ordinal(a_bits) - ordinal(b_bits))
    return np.where(nan16(a_bits, act) & nan16(b_bits, act), 0, d)


def nan16(bits: np.ndarray, act) -> np.ndarray:
    return np.isnan(as_f64(bits, act))


class Guarded:
    """An output buffer with GUARD canary bytes on each side (the scale-buffer overrun of flashinfer
    PR #6631, Test changes, showed up only much later; a canary shows it at once)."""

    def __init__(self, nbytes: int, device, dtype=torch.uint8, shape=None):
        self.n = nbytes
        self.buf = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device=device)
        self.view = self.buf[GUARD:GUARD + nbytes].view(dtype)
        if shape is not None:
            self.view = self.view.view(shape)

    def guards_intact(self) -> bool:
        b = self.buf.cpu().numpy()
        return bool(np.all(b[:GUARD] == CANARY) and np.all(b[GUARD + self.n:] == CANARY))

    def payload(self) -> np.ndarray:
        return self.buf[GUARD:GUARD + self.n].cpu().numpy()


def partials_of(case):
    import moe_finalize_residual_gb300 as mfr
    return [mfr.Partial(case.gemm2[r], case.perm[r], case.scale[r], case.shared[r]) for r in range(case.R)]


@dataclasses.dataclass
class Result:
    residual_out: np.ndarray
    norm_out: np.ndarray
    quant_out: np.ndarray | None
    sf_out: np.ndarray | None
    guards_ok: bool
    sf_raw: Guarded | None = None


def run(case, kernel="auto", pdl=True, routing_ready=False, quant="none", qscale=None, sf_layout="row_major",
        residual_out=True, norm_out=True, stream=None, extra_flags=0) -> Result:
    """Run the library on a device-resident case with canary-guarded outputs."""
    import moe_finalize_residual_gb300 as mfr
    dev = case.device
    T, H = case.T, case.H
    act = case.act_dtype
    ro = Guarded(T * H * 2, dev, act, (T, H)) if residual_out else None
    no = Guarded(T * H * 2, dev, act, (T, H)) if norm_out else None
    qo = sf = None
    if quant != "none":
        qo = Guarded(mfr.moe_finalize_quant_bytes(T, H, quant), dev)
        if quant == "nvfp4":
            sf = Guarded(mfr.moe_finalize_sf_bytes(T, H, sf_layout), dev)
    mfr.moe_finalize_fused(partials_of(case), case.residual, case.gamma, routed_scaling_factor=case.rsf,
                           eps=case.eps, residual_out=None if ro is None else ro.view,
                           norm_out=None if no is None else no.view, want_residual_out=False, want_norm_out=False,
                           quant_mode=quant, quant_scale=qscale, sf_layout=sf_layout,
                           quant_out=None if qo is None else qo.view, sf_out=None if sf is None else sf.view,
                           pdl=pdl, routing_ready=routing_ready, kernel=kernel, stream=stream,
                           extra_flags=extra_flags)
    torch.cuda.synchronize()
    ok = all(g.guards_intact() for g in (ro, no, qo, sf) if g is not None)
    return Result(bits16(ro.view) if ro else None, bits16(no.view) if no else None,
                  qo.payload() if qo else None, sf.payload() if sf else None, ok, sf)


def check_against_oracle(case_cpu, res: Result, want=None, mae_slack=0.01, tokens=None):
    """residual_out bit-exact; norm_out within 1 ulp; MAE vs FP64 no worse than the oracle's (+slack)."""
    want = want if want is not None else oracle.finalize(case_cpu)
    act = case_cpu.act_dtype
    got_ro, got_no = res.residual_out, res.norm_out
    if tokens is not None:
        got_ro = got_ro[tokens]
        got_no = got_no[tokens]
    if got_ro is not None:
        w = want["residual_out"]
        same = (got_ro == w) | (nan16(got_ro, act) & nan16(w, act))
        assert same.all(), f"residual_out: {np.count_nonzero(~same)} of {same.size} elements differ"
    if got_no is not None:
        d = ulp_distance(got_no, want["norm_out"], act)
        assert d.max() <= 1, f"norm_out: max {d.max()} ulp; {np.count_nonzero(d > 1)} elements beyond 1 ulp"
        ref_res, ref_norm = oracle.finalize_fp64(case_cpu)
        fin = np.isfinite(ref_norm)
        if fin.any():
            mae_k = np.abs(as_f64(got_no, act) - ref_norm)[fin].mean()
            mae_o = np.abs(as_f64(want["norm_out"], act) - ref_norm)[fin].mean()
            assert mae_k <= mae_o * (1 + mae_slack) + 1e-12, (mae_k, mae_o)
    return want


def subcase(case, tokens) -> synth.Case:
    """A CPU problem holding only the given tokens of a (device) case, with the GEMM2 rows they read
    gathered into compact arrays and their indices remapped; out-of-range indices stay out of range."""
    tok = torch.as_tensor(tokens, dtype=torch.long, device=case.device)
    gemm2, perm, scale, shared = [], [], [], []
    for r in range(case.R):
        p = case.perm[r][tok].long()
        rows = case.gemm2[r].shape[0]
        valid = (p >= 0) & (p < rows)
        used = torch.unique(p[valid])
        remap = torch.full((rows,), -1, dtype=torch.long, device=case.device)
        remap[used] = torch.arange(used.numel(), device=case.device)
        newp = torch.where(valid, remap[p.clamp(0, rows - 1)], torch.full_like(p, -1))
        gemm2.append(case.gemm2[r][used].cpu())
        perm.append(newp.to(torch.int32).cpu())
        scale.append(None if case.scale[r] is None else case.scale[r][tok].cpu())
        shared.append(None if case.shared[r] is None else case.shared[r][tok].cpu())
    return dataclasses.replace(case, name=case.name + "-sub", T=len(tokens), gemm2=gemm2, perm=perm, scale=scale,
                               shared=shared, expert=[torch.zeros(0)] * case.R,
                               residual=case.residual[tok].cpu(), gamma=case.gamma.cpu())


def quant_scale_for(norm_bits: np.ndarray, act, quant: str) -> float:
    """Per-tensor scale mapping the largest |norm_out| to the top of the format: 448 for FP8,
    448 * 6 for the NVFP4 global scale."""
    amax = float(np.nanmax(np.abs(as_f64(norm_bits, act))))
    amax = amax if amax > 0 else 1.0
    return 448.0 / amax if quant == "fp8" else 448.0 * 6.0 / amax


def check_quant(res: Result, act, quant: str, qscale: float, sf_layout: str, T: int, H: int, want_norm=None):
    """Quantised bytes must equal the oracle's quantiser applied to the kernel's own norm_out, exactly;
    against the full oracle they may differ only in blocks whose norm_out differs."""
    lay = oracle.SF_ROW_MAJOR if sf_layout == "row_major" else oracle.SF_SWIZZLED_128x4
    qm = oracle.QUANT_FP8 if quant == "fp8" else oracle.QUANT_NVFP4
    q_own, sf_own = oracle.quantize(res.norm_out, act, qm, qscale, lay)
    got_q = res.quant_out.reshape(q_own.shape)
    assert np.array_equal(got_q, q_own), f"{quant}: {np.count_nonzero(got_q != q_own)} bytes differ"
    if quant == "nvfp4":
        n = oracle.sf_bytes(T, H, lay)
        written = np.zeros(n, dtype=bool)
        written[oracle.sf_offsets(T, H, lay).reshape(-1)] = True
        assert np.array_equal(res.sf_out[written], sf_own[written]), "block scales differ"
        assert np.all(res.sf_out[~written] == CANARY), "padding bytes of the scale buffer were written"
    if want_norm is not None:
        q_full, _ = oracle.quantize(want_norm, act, qm, qscale, lay)
        if quant == "fp8":
            same_in = res.norm_out == want_norm
            assert np.array_equal(got_q[same_in], q_full[same_in])
        else:
            blk_same = (res.norm_out == want_norm).reshape(T, H // 16, 16).all(axis=2)
            got_b = got_q.reshape(T, H // 16, 8)
            ful_b = q_full.reshape(T, H // 16, 8)
            assert np.array_equal(got_b[blk_same], ful_b[blk_same])


def contraction_case(act, T: int = 64, H: int = 1024, R: int = 2) -> synth.Case:
    """A case that tells "acc times the factor, rounded, then plus the shared row" from one fused
    multiply-add: one route per token with scale 1 (so acc is the gathered row itself), a factor with a
    full 24-bit significand (so the FP32 product is inexact), shared rows equal to minus the product
    rounded to act (so the add cancels the leading bits and exposes the product's rounding), and a zero
    residual (so nothing later swamps that difference)."""
    c = synth.make_case("contract", T=T, H=H, K=1, R=R, E=8, act_dtype=act, rsf=float(np.float32(1.0 / 3.0)),
                        shared=True, gemm2_std=1.0)
    for r in range(R):
        c.scale[r] = torch.ones_like(c.scale[r])
        rows = c.gemm2[r].double()[c.perm[r][:, 0].long()]  # 16-bit x 24-bit product: exact in FP64
        c.shared[r] = (-(rows * c.rsf)).to(act)
    c.residual = torch.zeros_like(c.residual)
    return c
