"""Pins for the oracle's MX formats and quantiser (CPU only).

Each check compares the oracle with something other than itself: the OCP MX
v1.0 E2M1 table (golden file), torch's independent float8_e4m3fn /
float8_e8m0fnu codecs, numpy's round-half-even, or hand cases.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden_lines


def test_e2m1_table_matches_ocp_spec():
    for ln in golden_lines("e2m1_values.txt"):
        code, val = ln.split()
        got = oracle.e2m1_value(int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), (code, got, val)


def test_e4m3_all_codes_match_torch():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), (c, got, ref[c])


def test_e8m0_all_codes_match_torch():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    for c in range(256):
        got = oracle.e8m0_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])


def _block_with_scale0(value, fmt):
    # A block whose amax fixes the shared exponent at 0: [4, 8) for E2M1
    # (emax 2), [256, 512) for E4M3 (emax 8).
    anchor = 4.0 if fmt == oracle.FMT_E2M1 else 256.0
    v = np.zeros(32)
    v[0] = anchor
    v[1] = value
    return v


def _decode(code, fmt):
    return oracle.e2m1_value(code) if fmt == oracle.FMT_E2M1 else oracle.e4m3_value(code)


def test_quantizer_hand_cases():
    for ln in golden_lines("quantizer_hand_cases.txt"):
        f, v, exp = ln.split()
        fmt = oracle.FMT_E2M1 if f == "e2m1" else oracle.FMT_E4M3
        codes, sc = oracle.mx_quantize_block(_block_with_scale0(float(v), fmt), fmt)
        assert sc == 127, ln
        got = _decode(int(codes[1]), fmt)
        assert got == float(exp) and math.copysign(1, got) == math.copysign(1, float(exp)), (ln, got)


def _e2m1_round_numpy(q):
    """Independent E2M1 RNE: the grid has quantum 0.5 on [0,2), 1 on [2,4),
    2 on [4,6]; numpy's round() is half-to-even on the quantum count, and the
    even count is the even code on each sub-grid."""
    a = np.abs(q)
    r = np.where(a < 2, np.round(a / 0.5) * 0.5, np.where(a < 4, np.round(a), np.round(a / 2) * 2))
    return np.copysign(np.minimum(r, 6.0), q)


def test_e2m1_quantizer_matches_numpy_rounding():
    rng = np.random.default_rng(0)
    for trial in range(400):
        v = rng.normal(0, 1, 32) * (2.0 ** rng.integers(-20, 20))
        if trial % 5 == 0:  # exact ties on the grid after scaling
            v = rng.integers(-14, 15, 32) * 0.25 * (2.0 ** rng.integers(-5, 5))
        codes, sc = oracle.mx_quantize_block(v, oracle.FMT_E2M1)
        amax = np.max(np.abs(v))
        e = math.frexp(amax)[1] - 1 - 2 if amax > 0 else -127
        assert sc == e + 127
        q = v * 2.0 ** (-e)
        ref = _e2m1_round_numpy(q)
        got = np.array([oracle.e2m1_value(int(c)) for c in codes])
        np.testing.assert_array_equal(got, ref)
        np.testing.assert_array_equal(np.signbit(got), np.signbit(ref))


def test_e4m3_quantizer_matches_torch_rounding():
    # torch's fp32 -> float8_e4m3fn cast rounds to nearest even; values above
    # 448 become NaN there, so saturation is checked separately.
    rng = np.random.default_rng(1)
    for trial in range(300):
        v = (rng.normal(0, 1, 32) * (2.0 ** rng.integers(-30, 30))).astype(np.float32).astype(np.float64)
        if trial % 4 == 0:
            v[rng.integers(0, 32)] = 0.0
        codes, sc = oracle.mx_quantize_block(v, oracle.FMT_E4M3)
        amax = np.max(np.abs(v))
        e = math.frexp(amax)[1] - 1 - 8
        assert sc == e + 127
        q = torch.from_numpy(v * 2.0 ** (-e)).float()  # exact: power-of-two scaling of fp32 values
        sat = q.abs() > 448
        ref = q.clamp(-448, 448).to(torch.float8_e4m3fn)
        ref_codes = ref.view(torch.uint8).numpy()
        np.testing.assert_array_equal(codes[~sat.numpy()], ref_codes[~sat.numpy()])
        assert all(int(c) & 0x7F == 0x7E for c in codes[sat.numpy()])


def test_scale_exponent_edges():
    # amax exactly a power of two, just below it, zero, and tiny/huge blocks.
    for amax, fmt, expect in [(1.0, 1, 119), (np.nextafter(1.0, 0), 1, 118), (0.5, 0, 124), (6.0, 0, 127),
                              (8.0, 0, 128), (0.0, 0, 0), (0.0, 1, 0), (2.0 ** -140, 1, 0),
                              (2.0 ** 130, 0, 254)]:
        v = np.zeros(32)
        v[3] = amax
        _, sc = oracle.mx_quantize_block(v, fmt)
        assert sc == expect, (amax, fmt, sc)


def test_zero_block_keeps_signs():
    v = np.zeros(32)
    v[::2] = -0.0
    codes, sc = oracle.mx_quantize_block(v, oracle.FMT_E4M3)
    assert sc == 0
    assert all(c == (0x80 if i % 2 == 0 else 0) for i, c in enumerate(codes))


def test_bf16_rounding():
    # Values exactly representable in fp32: torch's fp32 -> bf16 cast (RNE) is
    # an independent reference.
    rng = np.random.default_rng(2)
    v = (rng.normal(0, 1, 5000) * 2.0 ** rng.integers(-60, 60, 5000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_rne(float(x)) for x in v], np.uint16)
    np.testing.assert_array_equal(got, ref)
    # One rounding from fp64: 1 + 2^-8 is a tie (-> 1.0); 1 + 2^-8 + 2^-40 is
    # above the tie (-> 1 + 2^-7), which a detour through fp32 would miss.
    assert oracle.bf16_rne(1 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_rne(1 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.bf16_rne(-3584.0) == 0xC560
    assert oracle.bf16_rne(-83.90625) == 0xC2A8  # -84.0


@pytest.mark.parametrize("rows,K", [(3, 64), (5, 512)])
def test_quantize_rows_consistent_with_block(rows, K):
    rng = np.random.default_rng(rows)
    w = rng.normal(0, 0.02, (rows, K)).astype(np.float32)
    codes, scales = oracle.quantize_mxfp4(w)
    for r in range(rows):
        for b in range(K // 32):
            c, s = oracle.mx_quantize_block(w[r, b * 32:(b + 1) * 32].astype(np.float64), oracle.FMT_E2M1)
            assert scales[r, b] == s
            packed = codes[r, b * 16:(b + 1) * 16]
            unpacked = np.stack([packed & 0xF, packed >> 4], 1).reshape(-1)  # element 2i in the low nibble
            np.testing.assert_array_equal(unpacked, c)
