"""Pins for the CPU oracle: each checks it against something other than itself.

* the error table printed in flashinfer PR #6631 (Description, "mean abs error vs FP64");
* an FP64 evaluation of the same formula, with a per-element bound derived from the round points;
* a dense, non-permuted brute force on tiny inputs (numpy, FP64);
* bit-exact invariants of the definition (masking, identity, re-permutation, scaling, sign);
* closed forms of RMSNorm;
* the number formats against torch's conversions and the format definitions;
* a hand-worked NVFP4 block and hand-worked SWIZZLED_128x4 offsets;
* mutants: copies of the oracle source with one plausible mistake must fail a pin.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def as_f64(bits, act=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(act).double().numpy()


def ulp_distance(a_bits, b_bits):
    """Ordinal distance between two arrays of 16-bit float bit patterns (+0 and -0 are equal)."""
    def ordinal(b):
        b = b.astype(np.int32)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(ordinal(a_bits) - ordinal(b_bits))


# --------------------------------------------------------------------------------------------
# The page's error table
# --------------------------------------------------------------------------------------------

def p1_errors(T, H):
    c = synth.make_p1_case(T, H)
    ref_res, ref_norm = oracle.finalize_fp64(c)
    o = oracle.finalize(c)
    s = oracle.finalize(c, mode=oracle.MODE_STEP_ROUNDED)
    floor = np.abs(torch.from_numpy(ref_res).bfloat16().double().numpy() - ref_res).mean()
    return dict(res=np.abs(as_f64(o["residual_out"]) - ref_res).mean(),
                norm=np.abs(as_f64(o["norm_out"]) - ref_norm).mean(),
                stock_res=np.abs(as_f64(s["residual_out"]) - ref_res).mean(),
                stock_norm=np.abs(as_f64(s["norm_out"]) - ref_norm).mean(),
                floor=floor)


def check_p1_table(errs):
    g = json.load(open(os.path.join(GOLDEN, "p1_error_table.json")))
    # The page prints two significant digits (three for norm_out); the sample adds a little noise.
    assert abs(errs["res"] - g["residual_out"]["this_pr"]) <= 0.10e-3, errs
    assert abs(errs["norm"] - g["norm_out"]["this_pr"]) <= 0.04e-3, errs
    assert abs(errs["floor"] - g["residual_out"]["bf16_floor"]) <= 0.10e-3, errs
    lo, hi = g["residual_out"]["stock"]
    assert lo - 0.15e-3 <= errs["stock_res"] <= hi + 0.15e-3, errs
    lo, hi = g["norm_out"]["stock"]
    assert lo - 0.06e-3 <= errs["stock_norm"] <= hi + 0.06e-3, errs


@pytest.mark.parametrize("H", [6144, 7168])
def test_p1_error_table(H):
    check_p1_table(p1_errors(16, H))


# --------------------------------------------------------------------------------------------
# FP64 evaluation with a per-element bound
# --------------------------------------------------------------------------------------------

U32 = 2.0 ** -24


def unit(act):
    return 2.0 ** -8 if act == torch.bfloat16 else 2.0 ** -11


def residual_bound(case, o):
    """|residual_out - exact| bound from the definition's round points (FP32 steps + three act roundings)."""
    ua = unit(case.act_dtype)
    T, H, K = case.T, case.H, case.K
    tot = np.zeros((T, H))
    psum = np.zeros((T, H))
    for r in range(case.R):
        g = case.gemm2[r].double().numpy()
        perm = case.perm[r].numpy()
        sc = case.scale[r].double().numpy() if case.scale[r] is not None else np.ones((T, K))
        mag = np.zeros((T, H))
        for t in range(T):
            for k in range(K):
                i = perm[t, k]
                if 0 <= i < g.shape[0]:
                    mag[t] += np.abs(sc[t, k] * g[i])
        mag *= abs(case.rsf)
        if case.shared[r] is not None:
            mag += np.abs(case.shared[r].double().numpy())
        tot += (K + 2) * 1.01 * U32 * mag + ua * (mag + 1e-30)   # FP32 chain + rounding of p_r
        psum += mag
    S = as_f64(o["routed"], case.act_dtype)
    ro = as_f64(o["residual_out"], case.act_dtype)
    tot += case.R * 1.01 * U32 * psum * (1 + ua)                  # FP32 rank sum
    tot += ua * np.abs(S) + ua * np.abs(ro) + U32 * np.abs(ro)     # S rounding, residual add, final rounding
    return tot + 2.0 ** -133


CASES = [
    lambda: synth.make_case("tiny", T=4, H=256, K=2, R=1, E=8),
    lambda: synth.make_case("dec", T=3, H=512, K=8, R=4, E=64, rsf=2.5, shared=True),
    lambda: synth.make_case("msk16", T=5, H=256, K=10, R=2, E=32, act_dtype=torch.float16,
                            scale_dtype=torch.float32, mask_quarter=True),
    lambda: synth.make_case("hk", T=2, H=128, K=22, R=1, E=64, scale_dtype=torch.float32),
    lambda: synth.make_p1_case(3, 384),
]


@pytest.mark.parametrize("make", CASES)
def test_oracle_within_fp64_bound(make):
    c = make()
    o = oracle.finalize(c)
    ref_res, ref_norm = oracle.finalize_fp64(c)
    ro = as_f64(o["residual_out"], c.act_dtype)
    bound = residual_bound(c, o)
    assert np.all(np.abs(ro - ref_res) <= bound), np.max(np.abs(ro - ref_res) / bound)
    # norm_out: the oracle's rounded x through an FP64 RMSNorm, rounded to act, within 1 ulp
    x = ro
    rstd = 1.0 / np.sqrt((x * x).mean(axis=1, keepdims=True) + c.eps)
    want = (x * rstd * c.gamma.double().numpy()).astype(np.float32)
    want_bits = (oracle.f32_to_bf16(want) if c.act_dtype == torch.bfloat16 else oracle.f32_to_fp16(want))
    assert ulp_distance(o["norm_out"], want_bits).max() <= 1
    # and the whole chain stays close to the exact result: first-order propagation of the
    # residual error through RMSNorm, plus the final rounding
    ua = unit(c.act_dtype)
    gam = np.abs(c.gamma.double().numpy())
    rstd_ref = 1.0 / np.sqrt((ref_res * ref_res).mean(axis=1, keepdims=True) + c.eps)
    d_rstd = np.abs(rstd - rstd_ref) + rstd * c.H * U32
    nb = 1.01 * ua * np.abs(ref_norm) + gam * (rstd_ref * bound + np.abs(x) * d_rstd) * 1.01 + 1e-30
    err = np.abs(as_f64(o["norm_out"], c.act_dtype) - ref_norm)
    assert np.all(err <= nb), float(np.max(err / nb))


# --------------------------------------------------------------------------------------------
# Dense brute force (no permutation) on tiny inputs
# --------------------------------------------------------------------------------------------

def dense_fp64(case):
    """Rebuild each expert's rows from the expert-sorted layout, then sum over all E experts with a
    dense [T, E] weight matrix (zero off the top-k).  Uses the routing (expert ids) and the sort
    definition, never the perm array."""
    T, H, K, E = case.T, case.H, case.K, case.E
    total = np.zeros((T, H))
    for r in range(case.R):
        ids = case.expert[r].numpy()
        g = case.gemm2[r].double().numpy()
        W = np.zeros((T, E))
        sc = case.scale[r].double().numpy() if case.scale[r] is not None else np.ones((T, K))
        Y = np.zeros((T, E, H))
        pos = 0
        for e in range(E):                       # expert-sorted: expert by expert, tokens in order
            for t in range(T):
                for k in range(K):
                    if ids[t, k] == e:
                        Y[t, e] = g[pos]
                        W[t, e] += sc[t, k]
                        pos += 1
        out = np.einsum("te,teh->th", W, Y) * case.rsf
        if case.shared[r] is not None:
            out += case.shared[r].double().numpy()
        total += out
    return total + case.residual.double().numpy()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dense_brute_force(seed):
    c = synth.make_case("dense", T=3, H=64, K=3, R=2, E=6, rsf=2.5, shared=True, seed_base=seed * 77)
    dense = dense_fp64(c)
    ref_res, _ = oracle.finalize_fp64(c)
    np.testing.assert_allclose(ref_res, dense, rtol=1e-12, atol=1e-12)
    o = oracle.finalize(c)
    assert np.all(np.abs(as_f64(o["residual_out"]) - dense) <= residual_bound(c, o))


# --------------------------------------------------------------------------------------------
# Bit-exact invariants of the definition
# --------------------------------------------------------------------------------------------

def base_case(**kw):
    args = dict(name="inv", T=6, H=128, K=6, R=3, E=16, rsf=2.5, shared=True)
    args.update(kw)
    return synth.make_case(**args)


def same(o1, o2, keys=("residual_out", "norm_out", "routed")):
    for k in keys:
        assert np.array_equal(o1[k], o2[k]), k


def test_masked_route_equals_deleted_route():
    c = base_case()
    t, k, r = 2, 3, 1
    masked = synth.Case(**{**c.__dict__})
    masked.perm = [p.clone() for p in c.perm]
    masked.gemm2 = [g.clone() for g in c.gemm2]
    row = int(masked.perm[r][t, k])
    masked.perm[r][t, k] = -1
    masked.gemm2[r][row] = float("nan")          # nothing behind a masked route may leak
    deleted = synth.Case(**{**c.__dict__})
    keep = [j for j in range(c.K) if j != k]
    # token t loses route k; other tokens keep all K routes, so pad them with a masked route instead
    perm = [p.clone() for p in c.perm]
    scale = [s.clone() for s in c.scale]
    for rr in range(c.R):
        perm[rr] = torch.cat([perm[rr], torch.full((c.T, 1), -1, dtype=torch.int32)], dim=1)
        scale[rr] = torch.cat([scale[rr], torch.zeros((c.T, 1), dtype=scale[rr].dtype)], dim=1)
    perm[r][t] = torch.cat([c.perm[r][t, keep], torch.tensor([-1, -1], dtype=torch.int32)])
    scale[r][t] = torch.cat([c.scale[r][t, keep], torch.zeros(2, dtype=c.scale[r].dtype)])
    deleted.perm, deleted.scale, deleted.K = perm, scale, c.K + 1
    om, od = oracle.finalize(masked), oracle.finalize(deleted)
    same(om, od)
    assert not np.isnan(as_f64(om["residual_out"])).any()


def test_out_of_range_index_is_skipped():
    c = base_case()
    a = synth.Case(**{**c.__dict__})
    a.perm = [p.clone() for p in c.perm]
    b = synth.Case(**{**c.__dict__})
    b.perm = [p.clone() for p in c.perm]
    a.perm[0][1, 2] = -1
    b.perm[0][1, 2] = c.gemm2[0].shape[0] + 5      # beyond the rows: also a skip
    same(oracle.finalize(a), oracle.finalize(b))


def test_single_route_identity():
    c = synth.make_case("id", T=4, H=256, K=1, R=1, E=8, scale_dtype=None, rsf=1.0)
    o = oracle.finalize(c)
    rows = c.gemm2[0][c.perm[0][:, 0].long()]
    assert np.array_equal(o["routed"], rows.view(torch.int16).numpy().view(np.uint16))


def test_repermutation_invariance():
    c = base_case()
    d = synth.Case(**{**c.__dict__})
    g = torch.Generator().manual_seed(5)
    d.gemm2, d.perm = [], []
    for r in range(c.R):
        n = c.gemm2[r].shape[0]
        pi = torch.randperm(n, generator=g)
        newg = torch.empty_like(c.gemm2[r])
        newg[pi] = c.gemm2[r]
        d.gemm2.append(newg)
        d.perm.append(pi[c.perm[r].long()].to(torch.int32))
    same(oracle.finalize(c), oracle.finalize(d))


def test_power_of_two_rescaling():
    c = base_case()
    d = synth.Case(**{**c.__dict__})
    d.scale = [s * 2 for s in c.scale]
    d.rsf = c.rsf / 2
    same(oracle.finalize(c), oracle.finalize(d))


def test_zero_shared_equals_no_shared():
    c = base_case()
    d = synth.Case(**{**c.__dict__})
    d.shared = [torch.zeros_like(s) for s in c.shared]
    e = synth.Case(**{**c.__dict__})
    e.shared = [None] * c.R
    same(oracle.finalize(d), oracle.finalize(e))


def test_all_masked_extra_partials_equal_single_partial():
    c = base_case(R=1)
    d = base_case(R=3)
    d.gemm2[0], d.perm[0], d.scale[0], d.shared[0] = c.gemm2[0], c.perm[0], c.scale[0], c.shared[0]
    d.residual, d.gamma = c.residual, c.gamma
    for r in (1, 2):
        d.perm[r] = torch.full_like(d.perm[r], -1)
        d.shared[r] = None
    same(oracle.finalize(c), oracle.finalize(d))


def test_sign_symmetry():
    c = base_case()
    d = synth.Case(**{**c.__dict__})
    d.gemm2 = [-g for g in c.gemm2]
    d.shared = [-s for s in c.shared]
    d.residual = -c.residual
    o1, o2 = oracle.finalize(c), oracle.finalize(d)
    for k in ("residual_out", "norm_out"):
        a, b = as_f64(o1[k]), as_f64(o2[k])
        assert np.array_equal(a, -b)


def test_rank_order_is_fixed():
    """Swapping two partials can change rounding only through the FP32 rank sum; the oracle sums in
    rank order 0..R-1, so reordering the partials may change bits but never by more than 1 ulp."""
    c = base_case(R=4)
    d = synth.Case(**{**c.__dict__})
    order = [3, 1, 2, 0]
    for f in ("gemm2", "perm", "scale", "shared"):
        setattr(d, f, [getattr(c, f)[i] for i in order])
    assert ulp_distance(oracle.finalize(c)["routed"], oracle.finalize(d)["routed"]).max() <= 1


# --------------------------------------------------------------------------------------------
# RMSNorm closed forms
# --------------------------------------------------------------------------------------------

def residual_only_case(residual, gamma, eps):
    """A case whose routed sum is exactly zero (all routes masked), so residual_out == residual."""
    T, H = residual.shape
    c = synth.make_case("ro", T=T, H=H, K=1, R=1, E=4, rsf=1.0)
    c.perm = [torch.full((T, 1), -1, dtype=torch.int32)]
    c.residual, c.gamma, c.eps = residual, gamma, eps
    return c


@pytest.mark.parametrize("cval", [0.003, 0.5, -3.0, 40.0])
def test_rmsnorm_constant_row(cval):
    H, eps = 512, 1e-5
    res = torch.full((2, H), cval).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(H, generator=torch.Generator().manual_seed(1))).to(torch.bfloat16)
    o = oracle.finalize(residual_only_case(res, gamma, eps))
    cb = float(res[0, 0])
    want = cb / np.sqrt(cb * cb + eps) * gamma.double().numpy()
    assert np.array_equal(as_f64(o["residual_out"][0]), res[0].double().numpy())
    want_bits = oracle.f32_to_bf16(want.astype(np.float32))
    assert ulp_distance(o["norm_out"][0], want_bits).max() <= 1


def test_rmsnorm_unit_rms_before_gamma():
    H = 4096
    g = torch.Generator().manual_seed(3)
    res = (torch.randn(8, H, generator=g) * 2).to(torch.bfloat16)
    o = oracle.finalize(residual_only_case(res, torch.ones(H, dtype=torch.bfloat16), 1e-6))
    y = as_f64(o["norm_out"])
    x = res.double().numpy()
    ms = (x * x).mean(axis=1)
    rms = np.sqrt((y * y).mean(axis=1))
    np.testing.assert_allclose(rms, np.sqrt(ms / (ms + 1e-6)), rtol=2e-3)


# --------------------------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------------------------

def strided_f32(stride=997):
    u = np.arange(0, 2 ** 32, stride, dtype=np.uint64).astype(np.uint32)
    extra = np.array([0x00000000, 0x80000000, 0x3F808000, 0x3F818000, 0x7F7FFFFF, 0x7F7F8000,
                      0x00000001, 0x807FFFFF, 0x477FF000, 0x477FE000, 0x33000000, 0x33000001],
                     dtype=np.uint32)
    return np.concatenate([u, extra]).view(np.float32)


def test_bf16_rounding_matches_torch():
    x = strided_f32()
    got = oracle.f32_to_bf16(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all(got[nan] & 0x7F)


def test_fp16_rounding_matches_torch():
    x = strided_f32()
    got = oracle.f32_to_fp16(x)
    want = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])


def test_fmaf_is_fused():
    a = float(np.float32(1 + 2.0 ** -12))
    fused = oracle.fmaf(a, a, -1.0)
    assert fused == 2.0 ** -11 + 2.0 ** -24          # exact product kept
    assert float(np.float32(np.float32(a) * np.float32(a)) - np.float32(1.0)) == 2.0 ** -11


def test_e4m3_definition():
    assert oracle.e4m3_to_f32(0x38) == 1.0
    assert oracle.e4m3_to_f32(0x7E) == 448.0
    assert oracle.e4m3_to_f32(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_f32(0x01) == 2.0 ** -9
    assert np.isnan(oracle.e4m3_to_f32(0x7F)) and np.isnan(oracle.e4m3_to_f32(0xFF))
    vals = np.array([oracle.e4m3_to_f32(c) for c in range(0x7F)], dtype=np.float64)
    assert np.all(np.diff(vals) > 0)
    codes = oracle.f32_to_e4m3(vals.astype(np.float32))
    assert np.array_equal(codes, np.arange(0x7F, dtype=np.uint8))
    # midpoints round to the even code
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    got = oracle.f32_to_e4m3(mids)
    lo = np.arange(0x7E)
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8))
    # saturation and NaN
    assert list(oracle.f32_to_e4m3(np.array([449, 500, 1e30, np.inf, -np.inf, np.nan], np.float32))) == \
        [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F]


def test_e4m3_matches_torch_in_range():
    x = strided_f32(stride=4099)
    x = x[np.isfinite(x) & (np.abs(x) < 464)]
    got = oracle.f32_to_e4m3(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_e2m1_definition():
    grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert [oracle.e2m1_to_f32(c) for c in range(8)] == grid
    assert [oracle.e2m1_to_f32(c | 8) for c in range(8)] == [-v for v in grid]
    assert list(oracle.f32_to_e2m1(np.array(grid, np.float32))) == list(range(8))
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    assert list(oracle.f32_to_e2m1(ties)) == [0, 2, 2, 4, 4, 6, 6]
    assert list(oracle.f32_to_e2m1(np.array([6.5, 100, np.inf, -7, -0.0, 0.2, -0.3], np.float32))) == \
        [7, 7, 7, 15, 8, 0, 9]


def test_nvfp4_hand_worked_block():
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_block.json")))
    b = g["block"]
    v = torch.tensor(b["values"], dtype=torch.float32).to(torch.bfloat16).view(1, 16)
    q, sf = oracle.quantize(v.view(torch.int16).numpy().view(np.uint16), torch.bfloat16,
                            oracle.QUANT_NVFP4, b["global_scale"])
    assert int(sf[0]) == b["sf"]
    assert list(q[0]) == b["bytes"]


def test_nvfp4_scale_roundtrip():
    """sf codes the block amax to within E4M3 rounding; every code lies within 6 after scaling."""
    gen = torch.Generator().manual_seed(9)
    x = (torch.randn(4, 256, generator=gen) * 3).to(torch.bfloat16)
    gs = 448 * 6 / float(x.abs().max())
    q, sf = oracle.quantize(x.view(torch.int16).numpy().view(np.uint16), torch.bfloat16, oracle.QUANT_NVFP4, gs)
    xb = x.double().numpy().reshape(4, 16, 16)
    amax = np.abs(xb).max(axis=2).reshape(-1)
    sfv = np.array([oracle.e4m3_to_f32(int(c)) for c in sf])
    np.testing.assert_allclose(sfv, amax / 6 * gs, rtol=2 ** -3)
    # decode and compare to the input: within half an E2M1 step of the block scale (plus SF rounding)
    lo, hi = q & 0xF, q >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(4, 16, 16)
    dec = np.vectorize(oracle.e2m1_to_f32)(codes) * (sfv.reshape(4, 16, 1) / gs)
    assert np.all(np.abs(dec - xb) <= (sfv.reshape(4, 16, 1) / gs) * 1.0 + 1e-6)


def test_fp8_quant_simple():
    x = torch.tensor([[1.0, -2.0, 0.5, 448.0, 1000.0, -0.0, 3.0, 0.001]], dtype=torch.bfloat16)
    q, _ = oracle.quantize(x.view(torch.int16).numpy().view(np.uint16), torch.bfloat16, oracle.QUANT_FP8, 1.0)
    want = oracle.f32_to_e4m3(x.float().numpy()[0])
    assert list(q[0]) == list(want)
    assert q[0][4] == 0x7E and q[0][5] == 0x80


def test_fp8_scaled_hand_worked():
    """The FP8 output applies the per-tensor scale as an encode scale, q = e4m3(v * s): blocks worked by
    hand from the OCP E4M3 definition with s = 0.75 and s = 448/3 (ties, subnormal ties, saturation after
    scaling, signed zero)."""
    g = json.load(open(os.path.join(GOLDEN, "fp8_scaled.json")))
    for case in g["cases"]:
        v = torch.tensor([case["values"]], dtype=torch.float32).to(torch.bfloat16)
        assert torch.equal(v.float(), torch.tensor([case["values"]])), "fixture values must be exact in bf16"
        q, _ = oracle.quantize(v.view(torch.int16).numpy().view(np.uint16), torch.bfloat16, oracle.QUANT_FP8,
                               case["scale"])
        assert list(q[0]) == case["bytes"], (case["scale"], list(q[0]))


@pytest.mark.parametrize("act", [torch.bfloat16, torch.float16])
def test_fp8_scaled_matches_torch(act):
    """e4m3 of the fp32 product v * s by torch's own conversion (products kept below 464, where torch's
    float8_e4m3fn conversion rounds like the saturating encoder), for a small scale and for 448 / amax."""
    gen = torch.Generator().manual_seed(21)
    x = (torch.randn(8, 512, generator=gen) * 2.5).to(act)
    amax = float(x.float().abs().max())
    for s in (0.37, 448.0 / amax, 3.0):
        s32 = float(np.float32(s))
        prod = x.float() * s32
        keep = prod.abs() < 464
        q, _ = oracle.quantize(x.view(torch.int16).numpy().view(np.uint16), act, oracle.QUANT_FP8, s32)
        want = prod.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert keep.float().mean() > 0.5
        assert np.array_equal(q[keep.numpy()], want[keep.numpy()]), s
        assert np.all(q[~keep.numpy()] & 0x7F == 0x7E)  # the rest saturates to +-448


def test_sf_layouts():
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_block.json")))["swizzled_128x4_offsets"]
    for m, k, off in g["pairs"]:
        assert oracle.sf_offset(m, k, g["H"], oracle.SF_SWIZZLED_128x4) == off
    for T, H in [(1, 16), (130, 272), (300, 7168), (128, 64)]:
        n = oracle.sf_bytes(T, H, oracle.SF_SWIZZLED_128x4)
        assert n == ((T + 127) // 128) * 128 * ((H // 16 + 3) // 4) * 4
        Tp, Cp = ((T + 127) // 128) * 128, ((H // 16 + 3) // 4) * 4
        offs = [oracle.sf_offset(m, k, Cp * 16, oracle.SF_SWIZZLED_128x4) for m in range(Tp) for k in range(Cp)] \
            if T * H <= 300 * 272 else None
        if offs is not None:
            assert sorted(offs) == list(range(Tp * Cp))        # a bijection onto the padded buffer
        assert oracle.sf_bytes(T, H, oracle.SF_ROW_MAJOR) == T * H // 16
        assert oracle.sf_offset(T - 1, H // 16 - 1, H, oracle.SF_ROW_MAJOR) == T * H // 16 - 1


# --------------------------------------------------------------------------------------------
# Mutants: one plausible mistake each, planted in a copy of the oracle; a pin must catch it
# --------------------------------------------------------------------------------------------

MUTANTS = {
    "p_r not rounded": ("s = s + act_round(acc, dt);", "s = s + acc;"),
    "rank sum not rounded": ("float S = act_round(s, dt);", "float S = s;"),
    "norm on unrounded residual": (
        "x[h] = (dt == OR_BF16) ? oracle_bf16_to_f32(ro) : oracle_fp16_to_f32(ro);", "x[h] = S + res;"),
    "factor dropped": ("acc = acc * a->rsf;", "acc = acc;"),
    "factor after shared": (
        "acc = acc * a->rsf;\n          if (P->shared) acc = acc + act_load(P->shared, (int64_t)t * H + h, dt);",
        "if (P->shared) acc = acc + act_load(P->shared, (int64_t)t * H + h, dt);\n          acc = acc * a->rsf;"),
    "shared subtracted": ("if (P->shared) acc = acc + act_load", "if (P->shared) acc = acc - act_load"),
    "scale of wrong route": (
        "float sc = P->scale ? act_load(P->scale, (int64_t)t * K + k, a->scale_dtype) : 1.0f;",
        "float sc = P->scale ? act_load(P->scale, (int64_t)t * K + (K - 1 - k), a->scale_dtype) : 1.0f;"),
    "eps dropped": ("float rstd = 1.0f / sqrtf(ms + a->eps);", "float rstd = 1.0f / sqrtf(ms);"),
    "mean over H-1": ("float ms = ss / (float)H;", "float ms = ss / (float)(H - 1);"),
    "gamma ignored": ("a->norm_out[(int64_t)t * H + h] = act_round_bits((x[h] * rstd) * g, dt);",
                      "a->norm_out[(int64_t)t * H + h] = act_round_bits((x[h] * rstd), dt);"),
    "masked route read": ("if (idx < 0 || (int64_t)idx >= P->rows) continue;            /* masked route */",
                          "if (idx < 0) idx = 0;"),
    "nibbles swapped": ("q[j] = (uint8_t)(lo | (hi << 4));", "q[j] = (uint8_t)(hi | (lo << 4));"),
    "fp8 scale ignored": ("float p = v * qscale;", "float p = v;"),
    "fp8 scale divides": ("float p = v * qscale;", "float p = v / qscale;"),
    "sf from unscaled amax": ("float sf_in = (amax / 6.0f) * qscale;", "float sf_in = amax * qscale;"),
    "swizzle rows swapped": ("return tile * 512 + (r % 32) * 16 + (r / 32) * 4 + (k % 4);",
                             "return tile * 512 + (r / 4) * 16 + (r % 4) * 4 + (k % 4);"),
}


def all_pins():
    """Run every pin that can catch an arithmetic mistake; return the names of those that fail."""
    failed = []
    checks = [
        ("p1 table", lambda: check_p1_table(p1_errors(4, 6144))),
        ("fp64 bound", lambda: [test_oracle_within_fp64_bound(m) for m in CASES]),
        ("dense", lambda: test_dense_brute_force(0)),
        ("masking", test_masked_route_equals_deleted_route),
        ("constant row", lambda: [test_rmsnorm_constant_row(c) for c in (0.003, 0.5)]),
        ("unit rms", test_rmsnorm_unit_rms_before_gamma),
        ("nvfp4 block", test_nvfp4_hand_worked_block),
        ("fp8 scaled", test_fp8_scaled_hand_worked),
        ("sf layout", test_sf_layouts),
    ]
    for name, fn in checks:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_contraction_case_is_discriminating(tmp_path):
    """The crafted case of the GPU contraction test must change under a fused shared-row step."""
    from helpers import contraction_case
    old = "acc = acc * a->rsf;\n          if (P->shared) acc = acc + act_load(P->shared, (int64_t)t * H + h, dt);"
    new = "acc = P->shared ? fmaf(acc, a->rsf, act_load(P->shared, (int64_t)t * H + h, dt)) : acc * a->rsf;"
    src = oracle.source()
    assert src.count(old) == 1
    path = oracle.build_variant(src.replace(old, new), str(tmp_path / "libfused.so"))
    for act in (torch.bfloat16, torch.float16):
        case = contraction_case(act)
        want = oracle.finalize(case)["residual_out"]
        with oracle.use_library(path):
            fused = oracle.finalize(case)["residual_out"]
        frac = np.mean(fused != want)
        assert frac > 0.05, f"{act}: only {frac:.4f} of the outputs tell the fused step apart"


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_is_caught(mutant, tmp_path):
    old, new = MUTANTS[mutant]
    src = oracle.source()
    assert src.count(old) == 1, f"mutation site not found: {old!r}"
    path = oracle.build_variant(src.replace(old, new), str(tmp_path / "libmutant.so"))
    with oracle.use_library(path):
        failed = all_pins()
    assert failed, f"no pin caught the mutant '{mutant}'"


@pytest.mark.parametrize("threads", [1, 3, 16])
def test_threaded_oracle_is_bit_identical(threads):
    # The host-core baseline runs the oracle over token ranges in parallel; every token must come out
    # exactly as the single-threaded run gives it (masked routes, fp16, more threads than tokens).
    c = synth.make_case("thr", T=7, H=256, K=6, R=2, E=16, act_dtype=torch.float16, mask_quarter=True,
                        scale_dtype=torch.float32)
    a = oracle.finalize(c)
    b = oracle.finalize_threads(c, threads)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    part = oracle.finalize_threads(c, threads, 2, 5)
    assert np.array_equal(part["norm_out"][2:5], a["norm_out"][2:5])
    assert not part["norm_out"][:2].any() and not part["norm_out"][5:].any()
