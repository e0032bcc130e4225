"""The roofline's numerator on the host: the bytes per call that the definition must move, which
bench.py divides by the measured time.  Each expected figure is written out from the shapes
(the four arrays per partial, residual, gamma and the outputs), not from the function under test."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

bench = pytest.importorskip("bench")


def _headline(T):
    return synth.make_case("bytes", T=T, **bench.HEADLINE)


def test_headline_bytes_written_out():
    T, H, K, R = 128, 6144, 8, 4
    routing = R * T * K * (4 + 2)         # int32 index + bf16 scale per route
    rows = R * T * K * H * 2              # every route valid in the decode workload
    shared = R * T * H * 2
    residual, gamma = T * H * 2, H * 2
    outputs = 2 * T * H * 2               # residual_out + norm_out
    want = routing + rows + shared + residual + gamma + outputs
    assert want == 61_378_560
    assert bench.algorithmic_bytes(_headline(T)) == want


def test_quantised_outputs_replace_norm_out_bytes():
    T, H = 16, 6144
    c = _headline(T)
    plain = bench.algorithmic_bytes(c)
    assert plain - bench.algorithmic_bytes(c, quant="fp8") == T * H * 2 - T * H
    assert plain - bench.algorithmic_bytes(c, quant="nvfp4") == T * H * 2 - (T * H // 2 + T * H // 16)


def test_finalize_only_counts_no_residual_or_norm():
    T, H, K, R = 4, 6144, 8, 4
    c = _headline(T)
    want = R * T * K * 6 + R * T * K * H * 2 + R * T * H * 2 + T * H * 2
    assert bench.algorithmic_bytes(c, finalize_only=True) == want


def test_masked_routes_move_no_row_bytes():
    c = synth.make_case("bytes", T=8, H=256, K=4, R=2, E=16, mask_quarter=True)
    full = synth.make_case("bytes", T=8, H=256, K=4, R=2, E=16)
    masked = sum(int((p < 0).sum()) for p in c.perm)
    assert masked > 0
    assert bench.algorithmic_bytes(full) - bench.algorithmic_bytes(c) == masked * 256 * 2
