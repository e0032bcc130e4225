"""Parity of the CUDA library (through its C ABI) with the CPU oracle, on every workload family.

residual_out must be bit-identical to the oracle; norm_out within 1 ulp of the activation type
(only the order of the RMS sum of squares differs); the mean absolute error of norm_out against an
FP64 evaluation no worse than the oracle's own (1% slack); quantised bytes bit-identical to the
oracle's quantiser applied to the kernel's own norm_out.  Every output sits between canary guards.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (CANARY, contraction_case, Guarded, nan16, as_f64, bits16, check_against_oracle, check_quant, partials_of,
                     quant_scale_for, run, subcase, ulp_distance)

pytestmark = pytest.mark.gpu
KERNELS = ["cluster", "stream", "bulk"]


def on_gpu(case):
    return case.to("cuda")


def check_case(case, kernel, **kw):
    res = run(on_gpu(case), kernel=kernel, **kw)
    assert res.guards_ok, "an output guard was overwritten"
    return res, check_against_oracle(case, res)


# --------------------------------------------------------------------------------------------
# Workload families
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("pdl", [True, False])
@pytest.mark.parametrize("kernel", KERNELS + ["auto"])
def test_tiny(kernel, pdl):
    check_case(next(synth.config_cases("tiny")), kernel, pdl=pdl)


@pytest.mark.parametrize("T", synth.CONFIGS["decode"]["Ts"])
@pytest.mark.parametrize("kernel", KERNELS)
def test_decode(T, kernel):
    check_case(next(synth.config_cases("decode", Ts=(T,))), kernel)


def _masked_cases():
    """The whole masked workload: T x top-k x activation type x partials x scale type (flashinfer PR #6631,
    Test changes: top_k 6/8/10, a quarter of the routes -1, fp16 and bf16, TP2 and TP4)."""
    out = []
    for case_T in synth.CONFIGS["masked"]["Ts"]:
        for K in (6, 8, 10):
            for act in (torch.float16, torch.bfloat16):
                for R in (2, 4):
                    for sdt in (torch.float32, torch.bfloat16):
                        out.append((case_T, K, act, R, sdt))
    return out


@pytest.mark.parametrize("T,K,act,R,sdt", _masked_cases())
def test_masked(T, K, act, R, sdt):
    c = dict(synth.CONFIGS["masked"])
    c.pop("Ts")
    case = synth.make_case(f"masked-T{T}", T=T, K=K, R=R, act_dtype=act, scale_dtype=sdt, **c)
    for kernel in KERNELS:
        res, _ = check_case(case, kernel)
        assert not np.isnan(as_f64(res.residual_out, act)).any(), "a NaN row behind a masked route leaked"


@pytest.mark.parametrize("T", synth.CONFIGS["highk"]["Ts"])
@pytest.mark.parametrize("shape", synth.HIGHK_SHAPES)
def test_highk(shape, T):
    H, E, K = shape
    c = dict(synth.CONFIGS["highk"])
    c.pop("Ts")
    case = synth.make_case(f"highk-T{T}", T=T, H=H, E=E, K=K, **c)
    for kernel in KERNELS:
        check_case(case, kernel)


# --------------------------------------------------------------------------------------------
# Quantised outputs
# --------------------------------------------------------------------------------------------

QUANTS = [("fp8", "row_major"), ("nvfp4", "row_major"), ("nvfp4", "swizzled_128x4")]


@pytest.mark.parametrize("quant,layout", QUANTS)
@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("act", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("T", [1, 37, 130])
def test_quant_small(T, act, kernel, quant, layout):
    case = synth.make_case("q", T=T, H=1024, K=8, R=2, E=64, act_dtype=act, rsf=2.5, shared=True)
    want = oracle.finalize(case)
    qs = quant_scale_for(want["norm_out"], act, quant)
    res = run(on_gpu(case), kernel=kernel, quant=quant, qscale=qs, sf_layout=layout)
    assert res.guards_ok
    check_against_oracle(case, res, want)
    check_quant(res, act, quant, qs, layout, T, case.H, want_norm=want["norm_out"])


@pytest.mark.parametrize("quant,layout", [("none", "row_major")] + QUANTS)
@pytest.mark.parametrize("H", [6144, 16400])
def test_bulk_several_tokens_per_cta(H, quant, layout):
    """The bulk kernel with two or three tokens per CTA, so each token's epilogue is written between the
    next token's stages from alternating residual_out buffers; whole-row passes (H=6144) and two ragged
    passes (H=16400); every output form; every token against the oracle."""
    import moe_finalize_residual_gb300 as mfr
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = 2 * sms + 37
    case = synth.make_case("bulkmt", T=T, H=H, K=4, R=2, E=32, rsf=2.5, shared=True, mask_quarter=True)
    g = on_gpu(case)
    plan = mfr.moe_finalize_plan(partials_of(g), g.residual, g.gamma, kernel="bulk")
    assert plan["kernel"] == "bulk" and plan["grid"] < T, plan
    assert (plan["chunk"] < H) == (H > 14336), plan
    want = oracle.finalize(case)
    qs = quant_scale_for(want["norm_out"], case.act_dtype, quant) if quant != "none" else None
    res = run(g, kernel="bulk", quant=quant, qscale=qs, sf_layout=layout)
    assert res.guards_ok
    check_against_oracle(case, res, want)
    if quant != "none":
        check_quant(res, case.act_dtype, quant, qs, layout, T, H, want_norm=want["norm_out"])


@pytest.mark.parametrize("quant,layout", QUANTS)
@pytest.mark.parametrize("kernel", KERNELS)
def test_quant_without_norm_out(kernel, quant, layout):
    """norm_out may be omitted when a quantised output is requested; the quantised bytes are then those
    of the oracle's norm_out wherever the kernel's would agree (checked here by a second run)."""
    case = synth.make_case("qn", T=20, H=2048, K=6, R=1, E=32, rsf=1.0)
    g = on_gpu(case)
    qs = 37.5
    full = run(g, kernel=kernel, quant=quant, qscale=qs, sf_layout=layout)
    only = run(g, kernel=kernel, quant=quant, qscale=qs, sf_layout=layout, norm_out=False, residual_out=False)
    assert only.guards_ok and full.guards_ok
    assert np.array_equal(full.quant_out, only.quant_out)
    if quant == "nvfp4":
        assert np.array_equal(full.sf_out, only.sf_out)


def _gamma_sweep_case(gamma_bits: np.ndarray, T=2):
    """Rows of +-1 with every route masked and eps = 0, so rstd = 1 exactly and norm_out == +-gamma:
    the quantiser then sees every chosen bf16 value."""
    H = gamma_bits.size
    case = synth.make_case("sweep", T=T, H=H, K=1, R=1, E=4, rsf=1.0)
    case.perm = [torch.full((T, 1), -1, dtype=torch.int32)]
    sign = torch.ones(T, H)
    sign[1::2] = -1
    case.residual = sign.to(torch.bfloat16)
    case.gamma = torch.from_numpy(gamma_bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    case.eps = 0.0
    return case


@pytest.mark.parametrize("scale", [1.0, 0.75, 448.0 / 3.0, 2.0 ** -7])
@pytest.mark.parametrize("quant", ["fp8", "nvfp4"])
def test_codec_sweep_all_bf16(quant, scale):
    """Every finite bf16 value passes through the kernel's FP8 / NVFP4 conversion and must encode as the
    oracle's software codec says (ties to even, saturation, signed zero, subnormals)."""
    allbits = np.arange(65536, dtype=np.uint32)
    finite = ((allbits & 0x7F80) != 0x7F80)
    vals = allbits[finite]
    vals = np.concatenate([vals, np.zeros((-vals.size) % 32768, dtype=np.uint32)])
    for chunk in vals.reshape(-1, 32768):
        case = _gamma_sweep_case(chunk)
        res = run(on_gpu(case), kernel="cluster", quant=quant, qscale=scale)
        want_norm = np.stack([chunk.astype(np.uint16), (chunk ^ 0x8000).astype(np.uint16)])
        assert np.array_equal(res.norm_out, want_norm)
        check_quant(res, torch.bfloat16, quant, scale, "row_major", 2, case.H)


# --------------------------------------------------------------------------------------------
# Full sizes: sampled tokens against the oracle
# --------------------------------------------------------------------------------------------

def _sample_tokens(T, n=40, seed=0):
    g = np.random.default_rng(seed)
    picks = {0, 1, T - 1, T // 2, 127 % T, 128 % T}
    picks.update(int(x) for x in g.choice(T, size=min(T, n), replace=False))
    return sorted(picks)


@pytest.mark.parametrize("H", [6144, 7168])
@pytest.mark.parametrize("T", [1024, 4096, 16384])
def test_bandwidth_sampled(T, H):
    c = dict(synth.CONFIGS["bandwidth"])
    c.pop("Ts")
    case = synth.make_case(f"bandwidth-H{H}-T{T}", T=T, H=H, device="cuda", **c)
    toks = _sample_tokens(T)
    sub = subcase(case, toks)
    want = oracle.finalize(sub)
    for kernel in ("auto", "stream", "bulk"):
        res = run(case, kernel=kernel)
        assert res.guards_ok
        check_against_oracle(sub, res, want, tokens=toks)
    # quantised variants at the same size; the global scale assumes |norm_out| <= 8, which holds for unit-
    # variance residuals with gamma near 1 (values beyond it saturate identically on both sides)
    for kernel, quant, layout, qs in (("auto", "fp8", "row_major", 448.0 / 8),
                                      ("auto", "nvfp4", "row_major", 448.0 * 6 / 8),
                                      ("auto", "nvfp4", "swizzled_128x4", 448.0 * 6 / 8),
                                      ("bulk", "fp8", "row_major", 448.0 / 8),
                                      ("bulk", "nvfp4", "swizzled_128x4", 448.0 * 6 / 8)):
        res = run(case, kernel=kernel, quant=quant, qscale=qs, sf_layout=layout)
        assert res.guards_ok
        check_against_oracle(sub, res, want, tokens=toks)
        lay = oracle.SF_ROW_MAJOR if layout == "row_major" else oracle.SF_SWIZZLED_128x4
        qm = oracle.QUANT_FP8 if quant == "fp8" else oracle.QUANT_NVFP4
        q_own, sf_own = oracle.quantize(res.norm_out[toks], case.act_dtype, qm, qs, oracle.SF_ROW_MAJOR)
        if quant == "fp8":
            assert np.array_equal(res.quant_out.reshape(T, H)[toks], q_own)
        else:
            assert np.array_equal(res.quant_out.reshape(T, H // 2)[toks], q_own)
            offs = oracle.sf_offsets(T, H, lay)[toks]
            assert np.array_equal(res.sf_out[offs.reshape(-1)], sf_own)
        del res
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------------------------
# Edge cases
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", KERNELS)
def test_empty_batch_writes_nothing(kernel):
    case = synth.make_case("e", T=3, H=256, K=2, R=1, E=8)
    g = on_gpu(case)
    import moe_finalize_residual_gb300 as mfr
    out = Guarded(3 * 256 * 2, "cuda", torch.bfloat16, (3, 256))
    empty = g.residual[:0]
    parts = [mfr.Partial(g.gemm2[0], g.perm[0][:0], g.scale[0][:0], None)]
    mfr.moe_finalize_fused(parts, empty, g.gamma, residual_out=out.view[:0], norm_out=out.view[:0], kernel=kernel)
    torch.cuda.synchronize()
    assert out.guards_intact() and np.all(out.payload() == CANARY)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("H", [8, 24, 776, 4104, 32768])
def test_ragged_and_extreme_hidden(H, kernel):
    """H not a multiple of any slice or chunk size, the smallest H and the largest."""
    T = 3 if H < 32768 else 2
    case = synth.make_case("rag", T=T, H=H, K=4, R=2, E=16, rsf=2.5, shared=True)
    check_case(case, kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_max_slots(kernel):
    """R = 8 partials of K = 64 routes each, every one with a shared row: 520 rows per token."""
    case = synth.make_case("max", T=5, H=2048, K=64, R=8, E=128, rsf=0.5, shared=True, scale_dtype=torch.float16)
    check_case(case, kernel)


@pytest.mark.parametrize("T,H,R,K,act", [(40, 6144, 4, 8, torch.bfloat16), (96, 6144, 4, 8, torch.float16),
                                          (200, 7168, 2, 10, torch.bfloat16), (512, 6144, 4, 8, torch.bfloat16),
                                          (300, 4096, 1, 32, torch.bfloat16), (64, 32768, 8, 4, torch.float16)])
def test_cluster_chunks(T, H, R, K, act):
    """The cluster kernel with several chunks per CTA (medium batches), sampled tokens at the larger sizes."""
    import moe_finalize_residual_gb300 as mfr
    case = synth.make_case("chunks", T=T, H=H, K=K, R=R, E=64, act_dtype=act, rsf=2.5, shared=True,
                           mask_quarter=True, device="cuda")
    plan = mfr.moe_finalize_plan(partials_of(case), case.residual, case.gamma, kernel="cluster")
    assert plan["kernel"] == "cluster" and plan["stages"] >= 1
    toks = _sample_tokens(T) if T > 64 else np.arange(T)
    sub = subcase(case, toks)
    res = run(case, kernel="cluster")
    assert res.guards_ok
    check_against_oracle(sub, res, oracle.finalize(sub), tokens=toks)


def test_cluster_plans_use_chunks():
    """Medium batches give fewer CTAs per token, each covering several chunks, in one wave."""
    import moe_finalize_residual_gb300 as mfr
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for T in (64, 128, 256, 512):
        case = synth.make_case("p", T=T, H=6144, K=8, R=4, E=64, shared=True, device="cuda")
        plan = mfr.moe_finalize_plan(partials_of(case), case.residual, case.gamma)
        assert plan["kernel"] == "cluster", plan
        assert plan["stages"] >= 2 and plan["cluster"] * plan["stages"] * plan["chunk"] >= 6144, plan
        assert plan["grid"] == T * plan["cluster"] and plan["grid"] <= max(2 * sms, T), plan


def test_cluster_cta_size_choice():
    """Multi-chunk plans take 384-thread CTAs when the busiest SM then issues fewer row loads (decode T=64
    on 152 SMs: 4 CTAs of 384 threads per token, two chunks each, against 3 of 512), and keep 512
    threads on a tie (T=128: 2 CTAs of 512 threads, three chunks)."""
    import moe_finalize_residual_gb300 as mfr
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected plans are those of a 152-SM GB300")
    for T, want in ((64, (384, 4, 2)), (128, (512, 2, 3))):
        case = synth.make_case("p", T=T, H=6144, K=8, R=4, E=64, shared=True, device="cuda")
        plan = mfr.moe_finalize_plan(partials_of(case), case.residual, case.gamma)
        assert (plan["block"], plan["cluster"], plan["stages"]) == want, plan


@pytest.mark.parametrize("kernel", KERNELS)
def test_single_route_identity(kernel):
    case = synth.make_case("id", T=9, H=512, K=1, R=1, E=8, scale_dtype=None, rsf=1.0)
    res, _ = check_case(case, kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_out_of_range_and_negative_indices(kernel):
    case = synth.make_case("oor", T=6, H=1024, K=8, R=3, E=32, rsf=2.5, shared=True)
    for r in range(case.R):
        p = case.perm[r].clone()
        rows = case.gemm2[r].shape[0]
        p[0, 0] = rows          # one past the end
        p[1, 3] = rows + 12345
        p[2, 7] = -1
        p[3, 1] = -7
        p[4, :] = -1            # a token with no valid route in this partial
        case.perm[r] = p
    res, _ = check_case(case, kernel)
    assert not np.isnan(as_f64(res.residual_out, case.act_dtype)).any()


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("act", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("T", [3, 64, 200])
def test_shared_step_rounds_product_first(kernel, act, T):
    """acc times the factor is rounded to FP32 before the shared row is added; a fused multiply-add
    there changes a tenth to a quarter of this crafted case's outputs."""
    check_case(contraction_case(act, T=T), kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_mixed_shared_and_missing_scales(kernel):
    case = synth.make_case("mix", T=7, H=1536, K=6, R=4, E=32, rsf=2.5, shared=True)
    case.shared[1] = None
    case.shared[3] = None
    case.scale[2] = None
    check_case(case, kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("act", [torch.float16, torch.bfloat16])
def test_overflow_and_cancellation(kernel, act):
    """Large rows that overflow fp16, and partials that cancel (the tight fixture asked for in the review
    of flashinfer PR #6631: accumulation in FP32 must be visible in the result)."""
    case = synth.make_case("big", T=4, H=512, K=8, R=4, E=16, act_dtype=act, rsf=2.5, shared=True,
                           gemm2_std=3000.0 if act == torch.float16 else 1e30)
    check_case(case, kernel)
    c2 = synth.make_case("cancel", T=4, H=512, K=8, R=2, E=16, act_dtype=act, rsf=1.0)
    c2.gemm2[1] = -c2.gemm2[0]
    c2.perm[1] = c2.perm[0].clone()
    c2.scale[1] = c2.scale[0].clone()
    res, want = check_case(c2, kernel)
    # p_1 = -p_0 exactly, so the routed sum is 0 and residual_out == residual
    assert np.array_equal(res.residual_out, bits16(c2.residual))


# --------------------------------------------------------------------------------------------
# Launch modes
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", KERNELS)
def test_pdl_on_off_bitwise_equal_over_many_routings(kernel):
    """flashinfer PR #6546, Description: outputs with PDL on are bitwise equal to PDL off over 900
    routings (1-16 tokens, top-8).  The same count here, also with the early routing read."""
    n = 0
    for seed in range(150):
        for T in (1, 2, 5, 8, 13, 16):
            case = on_gpu(synth.make_case("pdl", T=T, H=2048, K=8, R=2, E=64, rsf=2.5, shared=True,
                                          seed_base=seed * 10_000))
            a = run(case, kernel=kernel, pdl=True)
            b = run(case, kernel=kernel, pdl=False)
            c = run(case, kernel=kernel, pdl=True, routing_ready=True)
            assert np.array_equal(a.residual_out, b.residual_out) and np.array_equal(a.norm_out, b.norm_out)
            assert np.array_equal(a.residual_out, c.residual_out) and np.array_equal(a.norm_out, c.norm_out)
            n += 1
    assert n == 900


@pytest.mark.parametrize("kernel", KERNELS)
def test_graph_replay_back_to_back(kernel):
    """flashinfer PR #6631 (walkthrough): capture 20 back-to-back launches, replay 50 times, check that
    it completes within 60 s and the result is right.  The deadline is a host loop on an event."""
    import moe_finalize_residual_gb300 as mfr
    case_cpu = synth.make_case("graph", T=64, H=6144, K=8, R=4, E=256, rsf=2.5, shared=True)
    g = on_gpu(case_cpu)
    ro = torch.empty_like(g.residual)
    no = torch.empty_like(g.residual)
    parts = partials_of(g)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            mfr.moe_finalize_fused(parts, g.residual, g.gamma, routed_scaling_factor=g.rsf, eps=g.eps,
                                   residual_out=ro, norm_out=no, kernel=kernel)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(20):
            mfr.moe_finalize_fused(parts, g.residual, g.gamma, routed_scaling_factor=g.rsf, eps=g.eps,
                                   residual_out=ro, norm_out=no, kernel=kernel)
    ro.zero_()
    ev = torch.cuda.Event()
    for _ in range(50):
        graph.replay()
    ev.record()
    deadline = time.time() + 60
    while not ev.query():
        assert time.time() < deadline, "graph replay did not finish within 60 s"
        time.sleep(0.001)
    from helpers import Result
    res = Result(bits16(ro), bits16(no), None, None, True)
    check_against_oracle(case_cpu, res)


def test_kernel_choice_and_plan():
    """The automatic choice follows the workload: the cluster kernel for small and medium batches and for
    small rows, the bulk-copy kernel once every SM streams several whole tokens of large rows -- for the
    decode rows (shared experts) and the bandwidth rows (none) alike."""
    import moe_finalize_residual_gb300 as mfr
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def plan(T, H, shared, R=4, K=8):
        c = synth.make_case("p", T=T, H=H, K=K, R=R, E=64, shared=shared, device="cuda")
        return mfr.moe_finalize_plan(partials_of(c), c.residual, c.gamma)
    p1 = plan(4, 6144, True)
    assert p1["kernel"] == "cluster" and p1["cluster"] >= 2 and p1["grid"] == 4 * p1["cluster"]
    for shared in (True, False):
        for H in (6144, 7168):
            assert plan(512, H, shared)["kernel"] == "cluster"
            pb = plan(6 * sms + 8, H, shared)
            assert pb["kernel"] == "bulk" and pb["grid"] == sms, pb
    assert plan(6 * sms + 8, 2048, False)["kernel"] == "cluster"  # 4 KB rows: cluster kernel


def test_gather_floor_copies_the_indexed_row():
    import moe_finalize_residual_gb300 as mfr
    rows = torch.arange(64 * 256, dtype=torch.int32, device="cuda").view(64, 256)  # 1 KB rows
    out = torch.zeros(128, dtype=torch.int32, device="cuda")
    for i in (0, 37, 63):
        mfr.moe_finalize_gather_floor_launch(torch.tensor([i], dtype=torch.int32, device="cuda"), rows, out)
        torch.cuda.synchronize()
        assert torch.equal(out, rows[i, :128])
    before = out.clone()
    mfr.moe_finalize_gather_floor_launch(torch.tensor([64], dtype=torch.int32, device="cuda"), rows, out)
    torch.cuda.synchronize()
    assert torch.equal(out, before)  # out of range: nothing written


def test_deterministic_repeats():
    case = on_gpu(synth.make_case("det", T=33, H=4096, K=8, R=4, E=64, rsf=2.5, shared=True))
    for kernel in KERNELS:
        a = run(case, kernel=kernel)
        for _ in range(3):
            b = run(case, kernel=kernel)
            assert np.array_equal(a.residual_out, b.residual_out) and np.array_equal(a.norm_out, b.norm_out)


def test_per_step_rounding_model_fails_parity():
    """Negative control: the old kernel's numerics (every step rounded to the activation type, as the
    pages describe) must not pass the parity check, so the check can tell the two apart."""
    case = synth.make_p1_case(8, 6144)
    res = run(on_gpu(case), kernel="cluster")
    stock = oracle.finalize(case, mode=oracle.MODE_STEP_ROUNDED)
    with pytest.raises(AssertionError):
        check_against_oracle(case, res, want=stock)
    check_against_oracle(case, res)


def test_invalid_arguments_write_nothing():
    import moe_finalize_residual_gb300 as mfr
    case = on_gpu(synth.make_case("bad", T=4, H=256, K=2, R=1, E=8))
    out = Guarded(4 * 256 * 2, "cuda", torch.bfloat16, (4, 256))
    parts = partials_of(case)
    with pytest.raises(mfr.MoEFinalizeError, match="sf_out"):
        _call_without_sf(mfr, parts, case, out)
    with pytest.raises(ValueError):
        mfr.moe_finalize_fused(parts, case.residual.cpu(), case.gamma, residual_out=out.view)
    # quantised buffers one byte short of what the call writes: refused before the launch
    short_q = torch.empty(4 * 256 // 2 - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError, match="quant_out"):
        mfr.moe_finalize_fused(parts, case.residual, case.gamma, residual_out=out.view, quant_mode="nvfp4",
                               quant_scale=1.0, quant_out=short_q)
    short_sf = torch.empty(mfr.moe_finalize_sf_bytes(4, 256, "swizzled_128x4") - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError, match="sf_out"):
        mfr.moe_finalize_fused(parts, case.residual, case.gamma, residual_out=out.view, quant_mode="nvfp4",
                               quant_scale=1.0, sf_layout="swizzled_128x4", sf_out=short_sf)
    torch.cuda.synchronize()
    assert out.guards_intact() and np.all(out.payload() == CANARY)


def _call_without_sf(mfr, parts, case, out):
    import ctypes
    a, keep = mfr._build_args(parts, case.residual, case.gamma, 1.0, 1e-6, out.view, None, 2,
                              torch.ones(1, device="cuda"), 0, torch.empty(512, dtype=torch.uint8, device="cuda"),
                              None, 1, 0, check=False)
    mfr._check(mfr.raw_library().moe_finalize_fused(ctypes.byref(a), None))


def test_no_wait_timed_out():
    import moe_finalize_residual_gb300 as mfr
    assert mfr.moe_finalize_read_timeouts() == 0


def test_exchange_wait_that_runs_out_is_counted():
    """Failure detection on the GPU without a fault: the test hook makes the cluster exchange barrier
    expect 4 bytes that no peer sends (a signal that never comes), so every warp's wait on it runs out
    after its limit (about 2 s), is counted, and the kernel returns.  The context stays usable: the sums
    had all landed, so the outputs still match the oracle, and a normal call afterwards counts nothing."""
    import moe_finalize_residual_gb300 as mfr
    assert mfr.moe_finalize_read_timeouts() == 0
    case = synth.make_case("timeout", T=2, H=6144, K=8, R=4, E=64, rsf=2.5, shared=True)
    g = on_gpu(case)
    plan = mfr.moe_finalize_plan(partials_of(g), g.residual, g.gamma, kernel="cluster")
    assert plan["kernel"] == "cluster" and plan["cluster"] > 1, plan
    t0 = time.monotonic()
    res = run(g, kernel="cluster", extra_flags=mfr.MFR_FLAG_TEST_EXCHANGE_TIMEOUT)
    elapsed = time.monotonic() - t0
    assert mfr.moe_finalize_read_timeouts() == plan["grid"] * (plan["block"] // 32)  # every warp of every CTA
    assert 1.0 < elapsed < 60.0, elapsed
    check_against_oracle(case, res)
    check_against_oracle(case, run(g, kernel="cluster"))
    assert mfr.moe_finalize_read_timeouts() == 0


@pytest.mark.parametrize("kernel", ["stream", "bulk"])
def test_stream_wait_that_runs_out_is_counted(kernel):
    """Failure detection in the streaming kernels, on the GPU without a fault: the test hook makes the
    end-of-token barrier (where the compute warps meet to add their sums of squares) expect one arrival
    more than its warps give, so each wait on it runs out after its limit (about 2 s), is counted, and
    the kernel returns early (the abort flag stops the other warps; every copy in flight lands before the
    CTA exits).  The context stays usable: a normal call afterwards matches the oracle and counts
    nothing.  At most one token per CTA (groups splitting a token's hidden dimension in the stream
    kernel) and several tokens per CTA."""
    import moe_finalize_residual_gb300 as mfr
    assert mfr.moe_finalize_read_timeouts() == 0
    for T, H in ((4, 1024), (400, 256)):
        case = synth.make_case("stream-timeout", T=T, H=H, K=8, R=2, E=64, rsf=2.5, shared=True)
        g = on_gpu(case)
        plan = mfr.moe_finalize_plan(partials_of(g), g.residual, g.gamma, kernel=kernel)
        assert plan["kernel"] == kernel, plan
        t0 = time.monotonic()
        res = run(g, kernel=kernel, extra_flags=mfr.MFR_FLAG_TEST_STREAM_TIMEOUT)
        elapsed = time.monotonic() - t0
        assert res.guards_ok
        assert mfr.moe_finalize_read_timeouts() > 0
        assert 1.0 < elapsed < 60.0, elapsed
        want = oracle.finalize(case)
        if T <= 152:  # one token per CTA: residual_out is written before the token's barrier
            assert np.array_equal(res.residual_out, want["residual_out"])
        check_against_oracle(case, run(g, kernel=kernel), want)
        assert mfr.moe_finalize_read_timeouts() == 0


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("H,E,K,R,shared,T", [(6144, 256, 8, 4, True, 1), (6144, 256, 8, 4, True, 16),
                                              (6144, 256, 8, 4, True, 128), (4096, 512, 32, 1, False, 16),
                                              (7168, 256, 10, 2, False, 64)])
def test_unfused_pair_matches_oracle(H, E, K, R, shared, T, kernel):
    """The unfused pair the benchmark times against the fused call (flashinfer PR #6631, Description:
    finalize, then a separate residual + RMSNorm kernel): finalize-only into S, then a second launch that
    reads S as the only row of a one-partial call with its route masked and factor 1 -- the bytes of a
    residual-RMSNorm kernel.  Both launches go out back to back with PDL; the pair must give the oracle's
    residual_out bit for bit and its norm_out within 1 ulp."""
    import moe_finalize_residual_gb300 as mfr
    case = synth.make_case("unfused", T=T, H=H, E=E, K=K, R=R, rsf=2.5, shared=shared,
                           scale_dtype=torch.float32 if R == 1 else torch.bfloat16, mask_quarter=not shared)
    g = on_gpu(case)
    s_out = torch.empty_like(g.residual)
    mfr.moe_finalize_routed(partials_of(g), routed_scaling_factor=g.rsf, out=s_out, kernel=kernel)
    masked = torch.full((T, 1), -1, dtype=torch.int32, device="cuda")
    second = synth.Case("second", T, H, 1, 1, 1, g.act_dtype, None, 1.0, g.eps, [g.gemm2[0][:1]], [masked], [None],
                        [s_out], [masked], g.residual, g.gamma)
    res = run(second, kernel=kernel)
    assert res.guards_ok
    check_against_oracle(case, res)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("T", [1, 16, 128, 600])
def test_residual_out_in_place(T, kernel):
    """residual_out may be the residual tensor itself (the usual in-place residual update): every element
    of residual is read by the same thread, before it writes that element of residual_out."""
    import moe_finalize_residual_gb300 as mfr
    case = synth.make_case("inplace", T=T, H=2048, K=8, R=2, E=64, rsf=2.5, shared=True)
    want = oracle.finalize(case)
    g = on_gpu(case)
    res_buf = g.residual.clone()
    norm = torch.empty_like(res_buf)
    mfr.moe_finalize_fused(partials_of(g), res_buf, g.gamma, routed_scaling_factor=g.rsf, eps=g.eps,
                           residual_out=res_buf, norm_out=norm, kernel=kernel)
    torch.cuda.synchronize()
    assert np.array_equal(bits16(res_buf), want["residual_out"])
    assert ulp_distance(bits16(norm), want["norm_out"]).max() <= 1


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("R", [2, 4])
def test_tp_one_shot_emulated_on_one_gpu(R, kernel):
    """The tensor-parallel path (moe_finalize_residual_gb300.tp) with its R ranks emulated in turn on the
    one GPU: rank r's finalize-only call gives its rounded partial p_r, the exchange hands every rank the
    slots p_0..p_{R-1} (gathered here without a collective), and every rank's fused call over the
    exchanged slots gives the oracle's R-partial residual_out bit for bit and its norm_out within 1 ulp."""
    import moe_finalize_residual_gb300 as mfr
    from moe_finalize_residual_gb300 import tp
    case = synth.make_case("tp", T=37, H=2048, K=8, R=R, E=64, rsf=2.5, shared=True, mask_quarter=True,
                           scale_dtype=torch.float32)
    g = on_gpu(case)
    parts = partials_of(g)
    slots = [mfr.moe_finalize_routed([parts[r]], routed_scaling_factor=g.rsf, kernel=kernel) for r in range(R)]
    want = oracle.finalize(case)
    for r in range(R):
        def exchange(p_r, group, r=r):
            assert torch.equal(p_r, slots[r])  # this rank's own row, finalized again by the protocol
            return slots
        ro, no, _, _ = tp.tp_finalize_fused(parts[r], g.residual, g.gamma, routed_scaling_factor=g.rsf, eps=g.eps,
                                            exchange=exchange, kernel=kernel)
        torch.cuda.synchronize()
        from helpers import Result
        check_against_oracle(case, Result(bits16(ro), bits16(no), None, None, True), want)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("quant,layout", QUANTS)
def test_tp_one_shot_quantised(quant, layout, kernel):
    """The tensor-parallel path with a quantised output: every rank's fused call over the exchanged slots
    gives the oracle's residual_out bit for bit, norm_out within 1 ulp, and the quantised bytes and block
    scales of the oracle's quantiser applied to its own norm_out."""
    import moe_finalize_residual_gb300 as mfr
    from moe_finalize_residual_gb300 import tp
    R = 2
    case = synth.make_case("tpq", T=21, H=1024, K=6, R=R, E=32, rsf=2.5, shared=True, mask_quarter=True)
    g = on_gpu(case)
    parts = partials_of(g)
    slots = [mfr.moe_finalize_routed([parts[r]], routed_scaling_factor=g.rsf, kernel=kernel) for r in range(R)]
    want = oracle.finalize(case)
    qs = quant_scale_for(want["norm_out"], case.act_dtype, quant)
    for r in range(R):
        ro, no, qo, sf = tp.tp_finalize_fused(parts[r], g.residual, g.gamma, routed_scaling_factor=g.rsf, eps=g.eps,
                                              exchange=lambda p_r, group: slots, kernel=kernel, quant_mode=quant,
                                              quant_scale=qs, sf_layout=layout)
        torch.cuda.synchronize()
        from helpers import Result
        res = Result(bits16(ro), bits16(no), qo.cpu().numpy(), None if sf is None else sf.cpu().numpy(), True)
        check_against_oracle(case, res, want)
        if quant == "fp8":
            check_quant(res, case.act_dtype, quant, qs, layout, case.T, case.H, want_norm=want["norm_out"])
        else:  # the binding zero-fills the padding of a scale buffer it allocates
            lay = oracle.SF_ROW_MAJOR if layout == "row_major" else oracle.SF_SWIZZLED_128x4
            q_own, sf_own = oracle.quantize(res.norm_out, case.act_dtype, oracle.QUANT_NVFP4, qs, lay)
            assert np.array_equal(res.quant_out.reshape(q_own.shape), q_own)
            written = np.zeros(oracle.sf_bytes(case.T, case.H, lay), dtype=bool)
            written[oracle.sf_offsets(case.T, case.H, lay).reshape(-1)] = True
            assert np.array_equal(res.sf_out[written], sf_own[written]) and np.all(res.sf_out[~written] == 0)


# ------------------------------------------------------------------------------------------------------
# Finalize-only mode: the rounded rank sum S (p_0 for one partial), no residual / RMSNorm / quant.

FIN_CASES = {
    "decode": dict(H=6144, K=8, R=4, E=64, rsf=2.5, shared=True),
    "masked": dict(H=7168, K=10, R=2, E=64, act_dtype=torch.float16, scale_dtype=torch.float32,
                   mask_quarter=True),
    "highk": dict(H=4096, K=32, R=1, E=512, scale_dtype=torch.float32),
    "single": dict(H=2048, K=6, R=1, E=32, rsf=2.5, shared=True),
}


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("T", [1, 37, 300])
@pytest.mark.parametrize("fam", sorted(FIN_CASES))
def test_finalize_only(fam, T, kernel):
    import moe_finalize_residual_gb300 as mfr
    case = synth.make_case(f"fin-{fam}", T=T, device="cuda", **FIN_CASES[fam])
    guard = Guarded(T * case.H * 2, "cuda", case.act_dtype, (T, case.H))
    out = mfr.moe_finalize_routed(partials_of(case), routed_scaling_factor=case.rsf, out=guard.view,
                                  kernel=kernel)
    torch.cuda.synchronize()
    assert guard.guards_intact(), "finalize_out guard overwritten"
    toks = _sample_tokens(T) if T > 64 else np.arange(T)
    sub = subcase(case, toks)
    want = oracle.finalize(sub)["routed"]
    got = bits16(out)[toks]
    same = (got == want) | (nan16(got, case.act_dtype) & nan16(want, case.act_dtype))
    assert same.all(), f"finalize_out: {np.count_nonzero(~same)} of {same.size} elements differ"


@pytest.mark.parametrize("kernel", KERNELS)
def test_finalize_only_large_batch(kernel):
    """Many tokens per CTA (both groups of the stream kernel, several chunks of the cluster kernel)."""
    import moe_finalize_residual_gb300 as mfr
    c = dict(synth.CONFIGS["bandwidth"])
    c.pop("Ts")
    case = synth.make_case("fin-bw", T=2048, H=7168, device="cuda", **c)
    out = mfr.moe_finalize_routed(partials_of(case), routed_scaling_factor=case.rsf, kernel=kernel)
    torch.cuda.synchronize()
    toks = _sample_tokens(2048)
    want = oracle.finalize(subcase(case, toks))["routed"]
    assert np.array_equal(bits16(out)[toks], want)


@pytest.mark.parametrize("kernel", KERNELS)
def test_finalize_out_with_fused_outputs(kernel):
    """finalize_out next to residual_out / norm_out: all three correct from one call."""
    import moe_finalize_residual_gb300 as mfr
    case = synth.make_case("fin-both", T=45, H=6144, K=8, R=4, E=64, rsf=2.5, shared=True, device="cuda")
    fin = torch.empty_like(case.residual)
    ro, no, _, _ = mfr.moe_finalize_fused(partials_of(case), case.residual, case.gamma,
                                          routed_scaling_factor=case.rsf, eps=case.eps, kernel=kernel,
                                          finalize_out=fin)
    torch.cuda.synchronize()
    want = oracle.finalize(case.to("cpu"))
    assert np.array_equal(bits16(fin), want["routed"])
    assert np.array_equal(bits16(ro), want["residual_out"])
    assert ulp_distance(bits16(no), want["norm_out"], case.act_dtype).max() <= 1


# --------------------------------------------------------------------------------------------
# Randomised shapes: many small problems drawn from a seeded generator, every kernel
# --------------------------------------------------------------------------------------------

def _random_shapes(n=36, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        K = int(rng.choice([1, 2, 3, 6, 8, 10, 16, 22, 32, 64]))
        R = int(rng.integers(1, 9))
        if K * R > 128:
            R = max(1, 128 // K)
        H = int(rng.choice([8, 16, 40, 256, 1000, 2048, 3584, 6144, 7168])) // 8 * 8
        if H % 16:
            quant = "none"
        else:
            quant = str(rng.choice(["none", "fp8", "nvfp4"]))
        out.append(dict(T=int(rng.integers(1, 70)), H=H, K=K, R=R, E=int(max(K, rng.integers(4, 80))),
                        act=[torch.bfloat16, torch.float16][int(rng.integers(2))],
                        sdt=[torch.float32, torch.bfloat16, torch.float16, None][int(rng.integers(4))],
                        shared=bool(rng.integers(2)), mask=bool(rng.integers(2)), rsf=float(rng.choice([1.0, 2.5, 0.75])),
                        quant=quant, layout=str(rng.choice(["row_major", "swizzled_128x4"])), seed=i))
    return out


@pytest.mark.parametrize("shape", _random_shapes(), ids=lambda s: f"T{s['T']}H{s['H']}K{s['K']}R{s['R']}{s['quant']}")
def test_random_shapes_all_kernels(shape):
    """Bit-exact residual_out, norm_out within 1 ulp and the oracle's quantiser on the kernel's own norm_out,
    for every kernel, on small problems of random shape, dtype, masking and output mode."""
    s = shape
    case = synth.make_case("rnd", T=s["T"], H=s["H"], K=s["K"], R=s["R"], E=s["E"], act_dtype=s["act"],
                           scale_dtype=s["sdt"], rsf=s["rsf"], shared=s["shared"], mask_quarter=s["mask"],
                           seed_base=70_000 + 131 * s["seed"])
    want = oracle.finalize(case)
    qs = quant_scale_for(want["norm_out"], s["act"], s["quant"]) if s["quant"] != "none" else None
    # A 1-ulp difference in one of a few hundred outputs moves the mean error by more than 1 %: small
    # problems get a wider margin on that one statistic (every element is still held to 1 ulp).
    slack = 0.01 if case.T * case.H >= 100_000 else 0.1
    for kernel in KERNELS + ["auto"]:
        res = run(on_gpu(case), kernel=kernel, quant=s["quant"], qscale=qs, sf_layout=s["layout"])
        assert res.guards_ok, kernel
        check_against_oracle(case, res, want, mae_slack=slack)
        if s["quant"] != "none":
            check_quant(res, s["act"], s["quant"], qs, s["layout"], case.T, case.H, want_norm=want["norm_out"])
    # finalize-only mode on the same problem: the rounded rank sum, bit for bit
    import moe_finalize_residual_gb300 as mfr
    g = on_gpu(case)
    for kernel in KERNELS + ["auto"]:
        guard = Guarded(case.T * case.H * 2, "cuda", case.act_dtype, (case.T, case.H))
        mfr.moe_finalize_routed(partials_of(g), routed_scaling_factor=case.rsf, out=guard.view, kernel=kernel)
        torch.cuda.synchronize()
        assert guard.guards_intact(), kernel
        got = bits16(guard.view)
        same = (got == want["routed"]) | (nan16(got, case.act_dtype) & nan16(want["routed"], case.act_dtype))
        assert same.all(), f"{kernel}: finalize_out differs in {np.count_nonzero(~same)} elements"
