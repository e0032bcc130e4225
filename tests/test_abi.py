"""Host-side checks of the C ABI that need no GPU: the library loads and exports every function the
header declares, the Python mirrors of the structs match the C layout, size queries agree with the
oracle's independent layout code, invalid arguments are rejected before any CUDA call, and the
package refuses to import without its library."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_finalize.h")


@pytest.fixture(scope="module")
def mfr():
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__._build_module().build()
    import moe_finalize_residual_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_finalize_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(mfr):
    names = declared_functions()
    assert len(names) >= 9, names
    lib = ctypes.CDLL(mfr.library_path())
    for n in names:
        assert hasattr(lib, n), f"{n} declared in moe_finalize.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", mfr.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (moe_finalize_\w+)", out))
    assert exported == set(names), exported ^ set(names)


def test_struct_layout_matches_header(tmp_path, mfr):
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stddef.h>
#include <stdio.h>
#include "moe_finalize.h"
#define F(s, m) printf(#s "." #m " %zu\n", offsetof(s, m))
int main(void) {
  printf("mfr_partial %zu\nmfr_args %zu\nmfr_plan %zu\n", sizeof(mfr_partial), sizeof(mfr_args), sizeof(mfr_plan));
  F(mfr_partial, gemm2_out); F(mfr_partial, num_rows); F(mfr_partial, perm_idx); F(mfr_partial, expert_scale);
  F(mfr_partial, shared_out);
  F(mfr_args, T); F(mfr_args, H); F(mfr_args, K); F(mfr_args, R); F(mfr_args, act_dtype); F(mfr_args, scale_dtype);
  F(mfr_args, routed_scaling_factor); F(mfr_args, eps); F(mfr_args, partials); F(mfr_args, residual);
  F(mfr_args, gamma); F(mfr_args, residual_out); F(mfr_args, norm_out); F(mfr_args, quant_mode);
  F(mfr_args, sf_layout); F(mfr_args, quant_scale); F(mfr_args, quant_out); F(mfr_args, sf_out);
  F(mfr_args, flags); F(mfr_args, kernel); F(mfr_args, finalize_out);
  F(mfr_plan, kernel); F(mfr_plan, grid); F(mfr_plan, cluster); F(mfr_plan, block); F(mfr_plan, smem_bytes);
  F(mfr_plan, chunk); F(mfr_plan, stages);
  printf("MFR_MAX_PARTIALS %d\nMFR_MAX_TOP_K %d\nMFR_ABI_VERSION %d\n", MFR_MAX_PARTIALS, MFR_MAX_TOP_K, MFR_ABI_VERSION);
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    c = dict(line.rsplit(" ", 1) for line in subprocess.check_output([str(exe)], text=True).splitlines())
    assert int(c["mfr_partial"]) == ctypes.sizeof(mfr._CPartial)
    assert int(c["mfr_args"]) == ctypes.sizeof(mfr._CArgs)
    assert int(c["mfr_plan"]) == ctypes.sizeof(mfr._CPlan)
    for cls, cname in ((mfr._CPartial, "mfr_partial"), (mfr._CArgs, "mfr_args"), (mfr._CPlan, "mfr_plan")):
        for fname, _ in cls._fields_:
            assert int(c[f"{cname}.{fname}"]) == getattr(cls, fname).offset, (cname, fname)
    assert int(c["MFR_ABI_VERSION"]) == mfr.moe_finalize_abi_version()


@pytest.mark.parametrize("T,H", [(1, 16), (4, 256), (127, 2048), (128, 7168), (129, 6144), (16384, 7168), (300, 272)])
def test_size_queries_match_oracle(mfr, T, H):
    for lay, olay in (("row_major", oracle.SF_ROW_MAJOR), ("swizzled_128x4", oracle.SF_SWIZZLED_128x4)):
        assert mfr.moe_finalize_sf_bytes(T, H, lay) == oracle.sf_bytes(T, H, olay)
    assert mfr.moe_finalize_quant_bytes(T, H, "fp8") == T * H
    assert mfr.moe_finalize_quant_bytes(T, H, "nvfp4") == T * H // 2
    assert mfr.moe_finalize_quant_bytes(T, H, "none") == 0


def _raw_args(mfr, **over):
    """A C argument block with plausible (never dereferenced) 256-byte-aligned fake pointers."""
    parts = (mfr._CPartial * 8)()
    for r in range(8):
        parts[r] = mfr._CPartial(0x10000 * (r + 1), 64, 0x900000 + 0x1000 * r, 0xA00000 + 0x1000 * r, None)
    a = mfr._CArgs()
    a.T, a.H, a.K, a.R = 8, 256, 8, 1
    a.act_dtype, a.scale_dtype = 0, 0
    a.routed_scaling_factor, a.eps = 1.0, 1e-6
    a.partials = ctypes.cast(parts, ctypes.POINTER(mfr._CPartial))
    a.residual, a.gamma, a.residual_out, a.norm_out = 0xB00000, 0xC00000, 0xD00000, 0xE00000
    a.quant_mode, a.sf_layout, a.kernel, a.flags = 0, 0, 0, 1
    for k, v in over.items():
        setattr(a, k, v)
    return a, parts


BAD = [
    dict(H=12), dict(H=0), dict(H=65536), dict(K=0), dict(K=65), dict(R=0), dict(R=9), dict(T=-1),
    dict(act_dtype=2), dict(scale_dtype=7), dict(quant_mode=3), dict(flags=8), dict(flags=1 | (1 << 28)),
    dict(kernel=4), dict(kernel=-1),
    dict(residual=None), dict(gamma=None), dict(residual=0xB00008), dict(norm_out=0xE00004),
    dict(residual_out=None, norm_out=None),
    dict(residual_out=None, norm_out=None, finalize_out=0xD00008),  # misaligned finalize_out
    dict(residual=None, finalize_out=0xF30000),  # residual may be absent only when finalize_out is the only output
    dict(quant_mode=1), dict(quant_mode=2, quant_scale=0xF00000, quant_out=0xF10000),
    dict(quant_mode=2, quant_scale=0xF00000, quant_out=0xF10000, sf_out=0xF20000, sf_layout=2),
    dict(quant_mode=2, quant_scale=0xF00000, quant_out=0xF10000, sf_out=0xF20000, H=264),
    dict(quant_mode=1, quant_scale=0xF00000, quant_out=0xF10004),  # FP8 output needs 8-byte alignment
    dict(quant_mode=2, quant_scale=0xF00000, quant_out=0xF10002, sf_out=0xF20000),  # NVFP4: 4-byte alignment
    dict(partials=None),
]


@pytest.mark.parametrize("over", BAD)
def test_invalid_arguments_rejected_on_host(mfr, over):
    lib = mfr.raw_library()
    if "partials" in over:
        a, keep = _raw_args(mfr)
        a.partials = None
    else:
        a, keep = _raw_args(mfr, **over)
    st = lib.moe_finalize_fused(ctypes.byref(a), None)
    assert st in (-1, -2), st
    assert lib.moe_finalize_last_error().decode() != ""
    plan = mfr._CPlan()
    assert lib.moe_finalize_plan(ctypes.byref(a), ctypes.byref(plan)) == st


def test_partial_pointer_checks(mfr):
    lib = mfr.raw_library()
    a, parts = _raw_args(mfr)
    parts[0].perm_idx = None
    assert lib.moe_finalize_fused(ctypes.byref(a), None) == -1
    a, parts = _raw_args(mfr)
    parts[0].gemm2_out = 0x10008
    assert lib.moe_finalize_fused(ctypes.byref(a), None) == -1
    a, parts = _raw_args(mfr)
    parts[0].num_rows = -3
    assert lib.moe_finalize_fused(ctypes.byref(a), None) == -1


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU error path")
def test_finalize_only_needs_no_residual_or_gamma(mfr):
    """With finalize_out the only output, residual and gamma may be NULL: validation passes and the call
    reaches the CUDA runtime (which reports no device here)."""
    a, keep = _raw_args(mfr, residual=None, gamma=None, residual_out=None, norm_out=None, finalize_out=0xF30000)
    assert mfr.raw_library().moe_finalize_fused(ctypes.byref(a), None) == -3


def test_empty_batch_is_a_no_op(mfr):
    a, keep = _raw_args(mfr, T=0)
    assert mfr.raw_library().moe_finalize_fused(ctypes.byref(a), None) == 0


def test_gather_floor_rejects_bad_buffers(mfr):
    lib = mfr.raw_library()
    assert lib.moe_finalize_gather_floor_launch(None, None, 1, 512, None, None, 0) == -1
    assert lib.moe_finalize_gather_floor_launch(0x1000, 0x1000, 1, 100, 0x1000, None, 0) == -1  # short rows
    assert lib.moe_finalize_gather_floor_launch(0x1000, 0x1008, 1, 512, 0x1000, None, 0) == -1  # misaligned


def test_status_strings(mfr):
    lib = mfr.raw_library()
    for s in (0, -1, -2, -3):
        assert lib.moe_finalize_status_string(s).decode().startswith("MFR_")


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_call_without_gpu_reports_cuda_error(mfr):
    a, keep = _raw_args(mfr)
    assert mfr.raw_library().moe_finalize_fused(ctypes.byref(a), None) == -3


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU error path")
def test_timeout_test_flag_passes_validation(mfr):
    """The failure-detection test hook is a known flag bit: validation accepts it (the call then reaches
    the CUDA runtime, which reports no device here)."""
    for flag in (mfr.MFR_FLAG_TEST_EXCHANGE_TIMEOUT, mfr.MFR_FLAG_TEST_STREAM_TIMEOUT):
        a, keep = _raw_args(mfr, flags=1 | flag)
        assert mfr.raw_library().moe_finalize_fused(ctypes.byref(a), None) == -3


def test_import_fails_loudly_without_library(tmp_path):
    pkg = tmp_path / "moe_finalize_residual_gb300"
    pkg.mkdir()
    src = os.path.join(ROOT, "moe_finalize_residual_gb300", "__init__.py")
    (pkg / "__init__.py").write_text(open(src).read())
    r = subprocess.run([sys.executable, "-c", "import moe_finalize_residual_gb300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "no CPU fallback" in r.stderr


def test_product_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "moe_finalize_residual_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b", text), f"{f} mentions the oracle"
    text = open(HEADER).read()
    assert "oracle" not in text
