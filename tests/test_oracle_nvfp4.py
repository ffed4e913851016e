"""Pins for the oracle's NVFP4 variant (CPU only): the FP4 path of "[SGLang]
CUTLASS MoE", section 6 -- E2M1 elements scaled in blocks of 16 by E4M3
scales, with an fp32 global scale per tensor (value = e2m1 * e4m3 / gs).

Hand-derived block cases (tests/golden/nvfp4_hand_cases.txt) fix the scale
rule, the element rounding (ties to even, saturation), the power-of-two
invariance of the global scale, the scale's saturation and underflow; the
block scale equals torch's round-to-nearest-even cast to float8_e4m3fn; the
reconstruction error stays within half an element step; a forward case worked
by hand fixes the dataflow (x and the weights quantised with their global
scales, the intermediate requantised with its own)."""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden_lines

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _cases():
    for ln in golden_lines("nvfp4_hand_cases.txt"):
        name, gs, vals, codes, sf = [f.strip() for f in ln.split("|")]
        yield name, float(gs), [float(v) for v in vals.split()], [int(c) for c in codes.split()], int(sf, 16)


@pytest.mark.parametrize("case", list(_cases()), ids=lambda c: c[0])
def test_block_hand_cases(case):
    name, gs, vals, codes, sf = case
    got, got_sf = oracle.nvfp4_quantize_block(np.asarray(vals, np.float32), gs)
    assert got_sf == sf, (name, got_sf)
    np.testing.assert_array_equal(got, codes)


def test_global_scale():
    assert oracle.nvfp4_global_scale(np.full((4, 8), 0.5, np.float32)) == 5376.0
    w = np.zeros((3, 16), np.float32)
    assert oracle.nvfp4_global_scale(w) == 1.0
    w[1, 5] = -3.0
    assert oracle.nvfp4_global_scale(w) == np.float32(2688.0) / np.float32(3.0)


def test_block_scale_is_torch_e4m3_rounding():
    # s = fp32(fp32(amax * gs) / 6) rounded to E4M3 by torch's own cast (no
    # saturation needed below 448)
    rng = np.random.default_rng(1)
    for _ in range(300):
        v = (rng.normal(0, 1, 16) * 2.0 ** rng.integers(-12, 12)).astype(np.float32)
        gs = np.float32(2.0 ** rng.uniform(-4, 8))
        amax = np.max(np.abs(v))
        s = np.float32(np.float32(amax * gs) / np.float32(6.0))
        if s > 448:
            continue
        _, sf = oracle.nvfp4_quantize_block(v, float(gs))
        want = torch.tensor([float(s)], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).item()
        assert sf == want, (s, sf, want)


def test_reconstruction_within_half_a_step():
    rng = np.random.default_rng(2)
    for _ in range(200):
        v = (rng.normal(0, 1, 16) * 2.0 ** rng.integers(-6, 6)).astype(np.float32)
        gs = float(np.float32(2.0 ** rng.uniform(0, 6)))
        codes, sf = oracle.nvfp4_quantize_block(v, gs)
        d = oracle.e4m3_value(sf)
        if d == 0:
            continue
        r = np.float32(np.float32(gs) / np.float32(d))
        q = np.abs(v.astype(np.float32) * r)
        dec = np.array([E2M1[c & 7] * (-1 if c & 8 else 1) for c in codes]) * d / gs
        for i in range(16):
            if q[i] >= 6:  # saturated: the largest element code
                assert codes[i] & 7 == 7
                continue
            k = np.searchsorted(E2M1, q[i])
            step = E2M1[min(k, 7)] - E2M1[max(k - 1, 0)] if k > 0 else 0.5
            assert abs(abs(dec[i]) - q[i] * d / gs) <= 0.5 * step * d / gs * (1 + 1e-6) + 1e-30, (v[i], dec[i])
        # the block scale is within half an E4M3 step of s = amax * gs / 6 (normal
        # binades: 3 mantissa bits; below 2^-6 the subnormal step 2^-9), so the
        # largest scaled element lands at 6 * s / dec(sf)
        sv = float(np.float32(np.float32(np.max(np.abs(v)) * np.float32(gs)) / np.float32(6.0)))
        if sv > 448.0:  # the scale saturates at the largest E4M3 value
            assert d == 448.0
            continue
        half = 2.0 ** (math.floor(math.log2(sv)) - 4) if sv >= 2.0 ** -6 else 2.0 ** -10
        assert abs(d - sv) <= half * (1 + 1e-9), (sv, d)
        assert np.max(q) <= 6.0 * sv / d * (1 + 1e-6)


def test_quantize_rows_pack_and_bf16_agree_with_blocks():
    rng = np.random.default_rng(3)
    w = rng.normal(0, 0.02, (3, 64)).astype(np.float32)
    gs = oracle.nvfp4_global_scale(w)
    codes, scales = oracle.quantize_nvfp4(w, gs)
    for r in range(3):
        for b in range(4):
            c, sf = oracle.nvfp4_quantize_block(w[r, 16 * b:16 * b + 16], gs)
            assert scales[r, b] == sf
            packed = codes[r, 8 * b:8 * b + 8]
            np.testing.assert_array_equal(packed & 0xF, c[0::2])
            np.testing.assert_array_equal(packed >> 4, c[1::2])
    xb = torch.from_numpy(w).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    xc, xs = oracle.quantize_nvfp4_bf16(bits, 448.0)
    xf = xb.float().numpy()
    for b in range(4):
        c, sf = oracle.nvfp4_quantize_block(xf[1, 16 * b:16 * b + 16], 448.0)
        np.testing.assert_array_equal(xc[1, 16 * b:16 * b + 16], c)
        assert xs[1, b] == sf


def _bf16_bits(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def test_forward_hand_case():
    # H = I = 32, one expert, k = 1 (routing weight 1), x == 1, every weight 0.5.
    # x with gs_x 448: s = 448 / 6 = 74.67 -> E4M3 72; r = 448 / 72 = 6.22 -> E2M1 6 (saturates), so
    #   x^ = 6 * 72 / 448 = 0.9642857.
    # weights: amax 0.5 -> gs = 5376, s = 448, r = 12, 0.5 * 12 = 6 -> w^ = 0.5 exactly.
    # G = U = 32 * 0.9642857 * 0.5 = 15.4286; h = silu(G) * U = 238.04.
    # h with gs_h 10.5: s = 238.04 * 10.5 / 6 = 416.6 -> E4M3 416; r = 10.5 / 416, h * r = 6.008 -> 6;
    #   h^ = 6 * 416 / 10.5 = 237.714.
    # Y = 32 * 237.714 * 0.5 = 3803.43 = out (bf16 3808).
    H = I = 32
    w1 = np.full((2 * I, H), 0.5, np.float32)
    w2 = np.full((H, I), 0.5, np.float32)
    g1, g2 = oracle.nvfp4_global_scale(w1), oracle.nvfp4_global_scale(w2)
    assert g1 == g2 == 5376.0
    c1, s1 = oracle.quantize_nvfp4(w1, g1)
    c2, s2 = oracle.quantize_nvfp4(w2, g2)
    r = oracle.forward_nvfp4(_bf16_bits([[1.0] * H]), np.zeros((1, 1), np.int32), np.ones((1, 1)),
                             np.zeros(1, np.int32), c1[None], s1[None], [g1], c2[None], s2[None], [g2],
                             x_gscale=448.0, h_gscale=10.5, H=H, I=I, E_global=1, E_local=1, expert_offset=0,
                             num_shared=0, want_act=True, want_xq=True)
    x_sf = 0x69  # E4M3 72 = 1.125 * 2^6
    assert oracle.e4m3_value(x_sf) == 72.0
    assert (r["xq"] == 7).all() and (r["xq_sf"] == x_sf).all()
    h_sf = 0x7D  # E4M3 416 = 1.625 * 2^8 (exponent field 8 + 7 = 15)
    assert oracle.e4m3_value(h_sf) == 416.0
    assert (r["act"] == 7).all() and (r["act_sf"] == h_sf).all()
    want = 32 * (6 * 416 / 10.5) * 0.5
    assert math.isclose(r["out_f64"][0, 0], want, rel_tol=1e-15)
    np.testing.assert_allclose(r["out_f64"], want, rtol=1e-15)
    assert (r["out_bf16"] == oracle.bf16_rne(3808.0)).all()


def test_forward_reduces_to_the_decoded_product():
    # an independent recomputation: decode the NVFP4 operands with torch's
    # float8 codec and numpy, multiply, requantise h with the oracle's block
    # rule, and compare the output within fp64 rounding
    rng = np.random.default_rng(4)
    H, I, E = 64, 32, 2
    w1 = rng.normal(0, 0.02, (E, 2 * I, H)).astype(np.float32)
    w2 = rng.normal(0, 0.02, (E, H, I)).astype(np.float32)
    q1 = [oracle.quantize_nvfp4(w1[e], oracle.nvfp4_global_scale(w1[e])) for e in range(E)]
    q2 = [oracle.quantize_nvfp4(w2[e], oracle.nvfp4_global_scale(w2[e])) for e in range(E)]
    g1 = [oracle.nvfp4_global_scale(w1[e]) for e in range(E)]
    g2 = [oracle.nvfp4_global_scale(w2[e]) for e in range(E)]
    x = torch.from_numpy(rng.normal(0, 1, (3, H)).astype(np.float32)).to(torch.bfloat16)
    xbits = x.view(torch.int16).numpy().view(np.uint16)
    ids = np.array([[0, 1], [1, 0], [1, 1]], np.int32)
    wts = np.array([[0.75, 0.25], [0.5, 0.5], [0.4, 0.6]])
    r = oracle.forward_nvfp4(xbits, ids, wts, np.arange(E, dtype=np.int32), np.stack([a for a, _ in q1]),
                             np.stack([b for _, b in q1]), g1, np.stack([a for a, _ in q2]),
                             np.stack([b for _, b in q2]), g2, x_gscale=448.0, h_gscale=500.0, H=H, I=I, E_global=E,
                             E_local=E, expert_offset=0, num_shared=0, want_act=True)
    f8 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()

    def dec(codes, scales, gs, K):
        lo, hi = codes & 0xF, codes >> 4
        c = np.stack([lo, hi], -1).reshape(codes.shape[0], K)
        mag = np.array(E2M1)[c & 7] * np.where(c & 8, -1.0, 1.0)
        return mag * np.repeat(f8[scales], 16, axis=1) / gs

    for t in range(3):
        xc, xs = oracle.quantize_nvfp4_bf16(xbits[t:t + 1], 448.0)
        xd = (np.array(E2M1)[xc[0] & 7] * np.where(xc[0] & 8, -1.0, 1.0)) * np.repeat(f8[xs[0]], 16) / 448.0
        out = np.zeros(H)
        for j in range(2):
            e = ids[t, j]
            W1 = dec(q1[e][0], q1[e][1], g1[e], H)
            gu = W1 @ xd
            h = (gu[:I] / (1 + np.exp(-gu[:I]))) * gu[I:]
            np.testing.assert_allclose(h.astype(np.float32), h, rtol=1e-7)
            hq = np.zeros(I)
            for b in range(I // 16):
                c, sf = oracle.nvfp4_quantize_block(h[16 * b:16 * b + 16].astype(np.float32), 500.0)
                assert (r["act"][t, j, 16 * b:16 * b + 16] == c).all() and r["act_sf"][t, j, b] == sf
                hq[16 * b:16 * b + 16] = np.array(E2M1)[c & 7] * np.where(c & 8, -1.0, 1.0) * f8[sf] / 500.0
            out += wts[t, j] * (dec(q2[e][0], q2[e][1], g2[e], I) @ hq)
        np.testing.assert_allclose(r["out_f64"][t], out, rtol=1e-12, atol=1e-15)
