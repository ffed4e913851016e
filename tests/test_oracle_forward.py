"""Pins for the oracle's layer forward (CPU only).

Hand-derived cases (tests/golden/forward_hand_cases.txt) fix every step of the
dataflow: x quantisation, gate/up order, SiLU, intermediate requantisation
with saturation, W2, the weighted sum over a token's experts and the bf16
rounding.  The structured (permutation) weights of case B make a transposed
operand or a shifted index give a different answer.  Further checks:
linearity in the routing weights, the expert-parallel slice sum, the shared
expert's additive contribution, and an independent re-computation of a small
random layer with torch's float8 codecs and numpy matmuls.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden_lines

H = I = 32


def _bf16_bits(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def _weights(w1_list, w2_list):
    """Quantise fp32 expert weights with the oracle: W1 [2I, H], W2 [H, I]."""
    q1 = [oracle.quantize_mxfp4(np.asarray(w, np.float32)) for w in w1_list]
    q2 = [oracle.quantize_mxfp4(np.asarray(w, np.float32)) for w in w2_list]
    return (np.stack([c for c, _ in q1]), np.stack([s for _, s in q1]),
            np.stack([c for c, _ in q2]), np.stack([s for _, s in q2]))


def _expert_structured():
    w1 = np.zeros((2 * I, H), np.float32)
    for r in range(I):
        w1[r, (r + 5) % H] = 2.0          # gate
        w1[I + r, (2 * r) % H] = 1.0      # up
    w2 = np.zeros((H, I), np.float32)
    for n in range(H):
        w2[n, (n + 3) % I] = 1.0
    return w1, w2


def _expert_const():
    w1 = np.concatenate([np.full((I, H), 0.25), np.full((I, H), -0.5)]).astype(np.float32)
    return w1, np.full((H, I), 0.125, np.float32)


def _run(x_rows, ids, w, experts):
    w1, w1s, w2, w2s = _weights([e[0] for e in experts], [e[1] for e in experts])
    E = len(experts)
    return oracle.forward(_bf16_bits(x_rows), np.asarray(ids, np.int32), np.asarray(w, np.float64),
                          np.arange(E, dtype=np.int32), w1, w1s, w2, w2s, H=H, I=I, E_global=E, E_local=E,
                          expert_offset=0, num_shared=0, want_act=True, want_xq=True)


def test_hand_case_A_saturating_requant():
    ones = (np.ones((2 * I, H), np.float32) * 0.5, np.ones((H, I), np.float32) * 0.5)
    r = _run([[1.0] * H], [[0]], [[1.0]], [ones, ones])
    assert (r["xq"] == 0x78).all() and (r["xq_sf"] == 119).all()
    assert (r["act"][0, 0] == 0x7E).all() and (r["act_sf"][0, 0] == 126).all()
    np.testing.assert_array_equal(r["out_f64"], np.full((1, H), 3584.0))
    assert (r["out_bf16"] == 0x4560).all()


def test_hand_case_B_structured_weights():
    x0 = [1.0 if h < 16 else 0.0 for h in range(H)]
    r = _run([x0, [0.5] * H], [[1], [0]], [[1.0], [1.0]], [_expert_const(), _expert_structured()])
    exp0 = np.zeros(H)
    exp0[[0, 1, 2, 3, 4, 29, 30, 31]] = 1.75
    np.testing.assert_array_equal(r["out_f64"][0], exp0)
    np.testing.assert_array_equal(r["out_f64"][1], np.full(H, -112.0))
    # intermediate of token 0: 8 saturated codes (1.75 = 448 * 2^-8), rest zero
    act = r["act"][0, 0]
    assert (act[:8] == 0x7E).all() and (act[8:] == 0).all() and r["act_sf"][0, 0, 0] == 119
    # token 1: every element saturates negative: -448 * 2^-4 = -28
    assert (r["act"][1, 0] == 0xFE).all() and r["act_sf"][1, 0, 0] == 123


def _run_act(x_rows, ids, w, experts, act, params):
    w1, w1s, w2, w2s = _weights([e[0] for e in experts], [e[1] for e in experts])
    E = len(experts)
    return oracle.forward(_bf16_bits(x_rows), np.asarray(ids, np.int32), np.asarray(w, np.float64),
                          np.arange(E, dtype=np.int32), w1, w1s, w2, w2s, H=H, I=I, E_global=E, E_local=E,
                          expert_offset=0, num_shared=0, want_act=True, activation=act, act_params=params)


@pytest.mark.parametrize("case,up,act,params,act_code,act_scale,out,out_bits", [
    ("D", 0.5, oracle.ACT_SWIGLU_CLAMP, (7.0,), 0x7C, 124, 768.0, 0x4440),
    ("E", -0.125, oracle.ACT_SWIGLU_CLAMP, (7.0,), 0xFE, 123, -448.0, 0xC3E0),
    ("F", 0.5, oracle.ACT_SITU, (4.0, 25.0), 0x7E, 124, 896.0, 0x4460),
])
def test_hand_cases_activation_variants(case, up, act, params, act_code, act_scale, out, out_bits):
    rows = {ln.split()[0]: ln.split() for ln in golden_lines("forward_hand_cases.txt")}
    assert rows[case][1] == "all" and float(rows[case][2]) == out and float(rows[case][4]) == out
    w1 = np.concatenate([np.full((I, H), 0.5), np.full((I, H), up)]).astype(np.float32)
    ex = (w1, np.full((H, I), 0.5, np.float32))
    r = _run_act([[1.0] * H], [[0]], [[1.0]], [ex, ex], act, params)
    assert (r["act"][0, 0] == act_code).all() and (r["act_sf"][0, 0] == act_scale).all()
    np.testing.assert_array_equal(r["out_f64"], np.full((1, H), out))
    assert (r["out_bf16"] == out_bits).all()


def _printed_situ_4_25(g, u):
    """The fixed-constant SiTU as the shape-templates page prints it (beta 4, lb 25)."""
    return 2.0 * math.tanh(g * 0.25) * (1.0 + math.tanh(g * 0.5)) * (25.0 * math.tanh(u * 0.04))


def test_situ_4_25_matches_the_printed_fixed_form():
    rng = np.random.default_rng(3)
    for g, u in list(rng.normal(0, 6, size=(200, 2))) + [(0.0, 1.0), (40.0, -60.0), (-40.0, 3.0)]:
        assert oracle.activation(oracle.ACT_SITU, (4.0, 25.0), g, u) == pytest.approx(_printed_situ_4_25(g, u),
                                                                                       rel=1e-12, abs=1e-12)


def test_activation_limits_and_symmetries():
    rng = np.random.default_rng(4)
    for g, u in rng.normal(0, 3, size=(200, 2)):
        sw = oracle.activation(oracle.ACT_SWIGLU, (), g, u)
        assert sw == pytest.approx(g / (1 + math.exp(-g)) * u, rel=1e-13, abs=1e-15)
        # unbounded constants reduce both variants to SwiGLU
        assert oracle.activation(oracle.ACT_SITU, (1e7, 1e7), g, u) == pytest.approx(sw, rel=1e-9, abs=1e-12)
        assert oracle.activation(oracle.ACT_SWIGLU_CLAMP, (1e9,), g, u) == sw
        # odd in the up projection
        assert oracle.activation(oracle.ACT_SITU, (2.0, 3.0), g, -u) == -oracle.activation(oracle.ACT_SITU,
                                                                                            (2.0, 3.0), g, u)
        # SiTU's factors are bounded by beta and lb
        assert abs(oracle.activation(oracle.ACT_SITU, (2.0, 3.0), g, u)) <= 2.0 * 3.0
    L = 1.5
    for g, u in [(0.3, -0.7), (-5.0, 1.0)]:  # inside the clamp (the gate is capped above only)
        assert oracle.activation(oracle.ACT_SWIGLU_CLAMP, (L,), g, u) == oracle.activation(oracle.ACT_SWIGLU, (), g, u)
    s = oracle.activation(oracle.ACT_SWIGLU, (), L, 1.0)  # silu(L)
    assert oracle.activation(oracle.ACT_SWIGLU_CLAMP, (L,), 9.0, 1.0) == s
    assert oracle.activation(oracle.ACT_SWIGLU_CLAMP, (L,), 9.0, 4.0) == pytest.approx(s * L, rel=1e-15)
    assert oracle.activation(oracle.ACT_SWIGLU_CLAMP, (L,), 9.0, -4.0) == pytest.approx(-s * L, rel=1e-15)
    assert oracle.activation(oracle.ACT_SWIGLU_CLAMP, (L,), -0.5, 4.0) == pytest.approx(
        oracle.activation(oracle.ACT_SWIGLU, (), -0.5, L), rel=1e-15)


def test_hand_case_C_weighted_sum():
    r = _run([[0.5] * H], [[0, 1]], [[0.75, 0.25]], [_expert_const(), _expert_structured()])
    np.testing.assert_array_equal(r["out_f64"][0], np.full(H, -83.90625))
    # each slot's row w * Y: the constant expert's h = silu(4) * -8 saturates
    # to -448 * 2^-4 = -28, Y = 32 * -28 * 0.125 = -112, times 0.75 -> -84; the
    # structured expert's Y = 0.375 (its one W2 entry per row picks one
    # intermediate code), times 0.25 -> 0.09375
    w = oracle.forward(_bf16_bits([[0.5] * H]), np.asarray([[0, 1]], np.int32), np.asarray([[0.75, 0.25]]),
                       np.arange(2, dtype=np.int32), *_weights([_expert_const()[0], _expert_structured()[0]],
                                                               [_expert_const()[1], _expert_structured()[1]]),
                       H=H, I=I, E_global=2, E_local=2, expert_offset=0, num_shared=0, want_y=True)["y_slot"]
    np.testing.assert_array_equal(w[0, 0], np.full(H, -84.0))
    np.testing.assert_array_equal(w[0, 1], np.full(H, 0.09375))
    assert (r["out_bf16"][0] == 0xC2A8).all()  # -84.0
    assert (r["act"][0, 1] == 0x7C).all() and r["act_sf"][0, 1, 0] == 117  # 384 = 1.5 * 2^8 -> 0x7C; * 2^-10 = 0.375


def _small_layer(seed=5, T=6, E=4, k=2, S=0, offset=0, E_local=None, Hh=64, Ii=64):
    cfg = synth.MoeConfig("t", seed, T=T, E_global=E, E_local=E if E_local is None else E_local,
                          expert_offset=offset, top_k=k, num_shared=S, hidden=Hh, inter=Ii, block_n=16)
    x = synth.x_host(cfg)
    lg = synth.logits_host(cfg)
    sl = synth.shared_logit_host(cfg)
    ids, w = oracle.route(lg, k, S, sl, 1.0)
    gids = cfg.global_ids
    q1 = oracle.quantize_mxfp4(synth.w1_host(cfg, gids).reshape(-1, Hh))
    q2 = oracle.quantize_mxfp4(synth.w2_host(cfg, gids).reshape(-1, Ii))
    n = gids.size
    wts = (q1[0].reshape(n, 2 * Ii, Hh // 2), q1[1].reshape(n, 2 * Ii, Hh // 32),
           q2[0].reshape(n, Hh, Ii // 2), q2[1].reshape(n, Hh, Ii // 32))
    return cfg, x, ids, w, wts


def _fwd(cfg, x, ids, w, wts):
    return oracle.forward(x, ids, w, np.arange(cfg.E_local + cfg.num_shared, dtype=np.int32), *wts,
                          H=cfg.hidden, I=cfg.inter, E_global=cfg.E_global, E_local=cfg.E_local,
                          expert_offset=cfg.expert_offset, num_shared=cfg.num_shared)


def test_linear_in_routing_weights():
    cfg, x, ids, w, wts = _small_layer()
    a = _fwd(cfg, x, ids, w, wts)["out_f64"]
    b = _fwd(cfg, x, ids, 2.0 * w, wts)["out_f64"]
    np.testing.assert_array_equal(b, 2.0 * a)  # power-of-two scaling is exact
    z = _fwd(cfg, x, ids, np.zeros_like(w), wts)["out_f64"]
    assert (z == 0).all()


def test_zero_w2_gives_zero_output():
    cfg, x, ids, w, wts = _small_layer()
    wts = (wts[0], wts[1], np.zeros_like(wts[2]), wts[3])
    assert (_fwd(cfg, x, ids, w, wts)["out_f64"] == 0).all()


def test_expert_parallel_slices_sum_to_full_layer():
    cfg, x, ids, w, wts = _small_layer(E=8, k=3, T=9)
    full = _fwd(cfg, x, ids, w, wts)["out_f64"]
    part = np.zeros_like(full)
    for off in (0, 4):
        c = cfg.replace(E_local=4, expert_offset=off)
        sl = tuple(a[off:off + 4] for a in wts)
        part += _fwd(c, x, ids, w, sl)["out_f64"]
    np.testing.assert_allclose(part, full, rtol=1e-12, atol=1e-12)


def test_slot_rows_sum_to_the_output_and_vanish_off_slice():
    cfg, x, ids, w, wts = _small_layer(E=8, k=3, T=9)
    c = cfg.replace(E_local=4, expert_offset=4)
    sl = tuple(a[4:8] for a in wts)
    r = oracle.forward(x, ids, w, np.arange(4, dtype=np.int32), *sl, H=c.hidden, I=c.inter, E_global=8, E_local=4,
                       expert_offset=4, num_shared=0, want_y=True)
    y = r["y_slot"]
    local = (ids >= 4) & (ids < 8)
    assert (y[~local] == 0).all() and (np.abs(y[local]).sum(axis=-1) > 0).all()
    acc = np.zeros_like(r["out_f64"])
    for j in range(ids.shape[1]):  # the oracle's own order: ascending j
        acc += y[:, j]
    np.testing.assert_array_equal(acc, r["out_f64"])


def test_shared_expert_adds_its_weighted_output():
    cfg, x, ids, w, wts = _small_layer(S=1)
    with_s = _fwd(cfg, x, ids, w, wts)["out_f64"]
    w_routed = w.copy()
    w_routed[:, -1] = 0.0
    routed_only = _fwd(cfg, x, ids, w_routed, wts)["out_f64"]
    # the shared slot alone, with weight 1, scaled by its routing weight
    w_shared = np.zeros_like(w)
    w_shared[:, -1] = 1.0
    y_s = _fwd(cfg, x, ids, w_shared, wts)["out_f64"]
    np.testing.assert_allclose(with_s, routed_only + w[:, -1:] * y_s, rtol=1e-12, atol=1e-12)


def _torch_mx_e4m3(v):
    """Independent MXFP8 quantiser: frexp scale + torch's RNE float8 cast."""
    v = np.asarray(v, np.float64).reshape(-1, 32)
    amax = np.abs(v).max(1)
    e = np.array([math.frexp(a)[1] - 1 - 8 if a > 0 else -127 for a in amax])
    q = torch.from_numpy(v * np.exp2(-e)[:, None]).float().clamp(-448, 448).to(torch.float8_e4m3fn)
    return (q.double().numpy() * np.exp2(e)[:, None]).reshape(-1)


def _np_e2m1_decode(codes, scales, K):
    lut = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])
    c = np.stack([codes & 0xF, codes >> 4], -1).reshape(codes.shape[0], K)
    s = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e8m0fnu).double().numpy()
    return lut[c] * np.repeat(s, 32, axis=1)


def test_independent_recomputation_small_layer():
    cfg, x, ids, w, wts = _small_layer(seed=11, T=5, E=4, k=2, S=1, Hh=96, Ii=64)
    ref = _fwd(cfg, x, ids, w, wts)["out_f64"]
    Hh, Ii = cfg.hidden, cfg.inter
    xf = synth.bf16_bits_to_f64(x)
    out = np.zeros((cfg.T, Hh))
    for t in range(cfg.T):
        xq = _torch_mx_e4m3(xf[t])
        for j in range(cfg.kp):
            gid = ids[t, j]
            e = gid if gid < cfg.E_global else cfg.E_local + gid - cfg.E_global
            W1 = _np_e2m1_decode(wts[0][e], wts[1][e], Hh)
            W2 = _np_e2m1_decode(wts[2][e], wts[3][e], Ii)
            gu = W1 @ xq
            h = gu[:Ii] / (1 + np.exp(-gu[:Ii])) * gu[Ii:]
            out[t] += w[t, j] * (W2 @ _torch_mx_e4m3(h))
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)
