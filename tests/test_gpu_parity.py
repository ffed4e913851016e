"""GPU path vs the oracle, through the C ABI (marked gpu).

Bars (from the layer's specification):
  - integer / byte results bit-exact: topk ids, expert counts and offsets,
    a_map, c_map, virtual experts, the MXFP8 bytes of x, the MXFP4 weight
    codes and scales;
  - topk weights: |w_gpu - w| <= 4e-6 * w + 1e-7 (fp32 exp / sum / divide);
  - intermediate act (FC1 -> activation -> MXFP8): identical codes except
    where fp32 tensor-core accumulation and fp64 differ across a rounding
    boundary: at most ACT_DIFF_FRACTION of the elements, each within one E4M3
    step of the larger of the two values, at the coarser of the two block
    scales (one scale step when the block exponent itself flips);
  - FC2 rows (w * Y of each routed slot whose intermediate equals the
    oracle's): relative L2 <= 1e-2 per row;
  - output bf16: relative L2 <= 1e-2 and max-abs <= 2e-2 against the fp64
    oracle.
Each layer check prints one "PARITY" line with the measured figures.
"""
import numpy as np
import pytest
import torch

import mxfp4_mixture_experts_02_gb300 as moe
import oracle
import synth
from moe_case import (E4M3_VALUES, OracleCase, bf16_bits, bf16_to_f64, dense_repeat_bound, device_inputs, device_weights,
                       rel_l2, shape_of, within_dense_repeat)

pytestmark = pytest.mark.gpu

SMALL = synth.MoeConfig("small", 7, T=48, E_global=64, E_local=64, expert_offset=0, top_k=4, num_shared=0,
                        hidden=1024, inter=256, block_n=32)

GRID = [
    SMALL.replace(T=1, block_n=16),
    SMALL.replace(T=7, block_n=32),
    SMALL.replace(T=48, block_n=16, num_shared=1, shared_scale=0.5),
    SMALL.replace(T=96, block_n=32, zipf_s=1.1),
    SMALL.replace(T=256, block_n=16, E_local=32, expert_offset=16),
    SMALL.replace(T=256, block_n=32, num_shared=1, zipf_s=1.1, hidden=1536, inter=384),
    SMALL.replace(T=200, block_n=128, top_k=8, num_shared=1, zipf_s=1.1),
    SMALL.replace(T=64, block_n=128, E_local=32, expert_offset=32, hidden=1536, inter=384),
    # the layer's own hidden size at small E: decode and 128-row tilings with
    # several items per CTA, full and cut 32-row slabs
    SMALL.replace(T=40, block_n=32, E_global=16, E_local=16, hidden=3584, inter=256),
    SMALL.replace(T=1200, block_n=128, E_global=8, E_local=8, top_k=2, hidden=3584, inter=128),
    synth.CONFIGS["tiny"],
    # FC1 activation variants (clamped SwiGLU, SiTU) with constants small
    # enough that the clamps and the tanh soft caps act on most elements
    SMALL.replace(T=48, block_n=32, activation=1, act_params=(0.75, 0.0)),
    SMALL.replace(T=96, block_n=16, num_shared=1, activation=2, act_params=(1.0, 0.5)),
    SMALL.replace(T=200, block_n=128, top_k=8, activation=1, act_params=(0.5, 0.0)),
    SMALL.replace(T=64, block_n=128, hidden=1536, inter=384, activation=2, act_params=(0.5, 0.25)),
    # past 512 tokens the decode tilings route, sort and quantise x in
    # separate launches
    SMALL.replace(T=600, block_n=32, num_shared=1, zipf_s=1.1),
]
FULL = [synth.CONFIGS[n] for n in ("decode_t32", "ep_slice_t64", "skewed_shared_t256", "prefill_t32768")]


def _cid(c):
    return "%s-T%d-B%d-E%d+%d-S%d-H%d-I%d-A%d" % (c.name, c.T, c.block_n, c.E_local, c.expert_offset,
                                                   c.num_shared, c.hidden, c.inter, c.activation)


_WCACHE = {}


def _weights(cfg):
    key = (cfg.seed, cfg.E_global, cfg.E_local, cfg.expert_offset, cfg.num_shared, cfg.hidden, cfg.inter)
    if key not in _WCACHE:
        _WCACHE.clear()
        _WCACHE[key] = device_weights(cfg)
    return _WCACHE[key]


def run_layer(cfg, T=None, path=moe.GEMM2_SPLIT):
    """The layer through moe_layer.  By default on the split GEMM2 path, whose
    FC2 writes the routed rows these tests compare (the dense path, which
    reduces them into the output instead, is tested in test_gpu_gemm2_gate.py)."""
    shape = shape_of(cfg, T)
    wts = _weights(cfg)
    x, logits, sl = device_inputs(cfg, T=shape.T)
    ws = moe.workspace(shape)
    moe.moe_set_gemm2_path(path)
    try:
        out, ids, w = moe.moe_layer(shape, logits, sl, x, wts, ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_gemm2_path(moe.GEMM2_AUTO)
    status = moe.moe_get_status(ws)
    return shape, ws, out, ids, w, status


def tile_scale_index(B, K, lane_major=False):
    """Byte offset inside a virtual expert's tile scale block of tile row i and
    K-block b.  Chunk-major (the intermediate's act_sf): per 128-K chunk a
    512-byte block, (i % 32) * 16 + (i / 32) * 4 + b % 4.  Lane-major (x at
    128-row tiles): the same 16-byte cells ordered by lane, then chunk:
    ((i % 32) * (K / 128) + b / 4) * 16 + (i / 32) * 4 + b % 4."""
    i = np.arange(B)[:, None]
    b = np.arange(K // 32)[None, :]
    if lane_major:
        return ((i % 32) * (K // 128) + b // 4) * 16 + (i // 32) * 4 + (b % 4)
    return (b // 4) * 512 + (i % 32) * 16 + (i // 32) * 4 + (b % 4)


def tile_scales_of_rows(sf_view, vinfo, num_v, K, rows, lane_major=False):
    """E8M0 scales [len(rows), K/32] of the given expert rows, read from the
    tile layout (only the virtual experts holding those rows leave the GPU)."""
    rows = np.asarray(rows, np.int64)
    firsts = vinfo[:num_v, 1].astype(np.int64)
    vs = np.searchsorted(firsts, rows, side="right") - 1  # first rows ascend with v
    idx = tile_scale_index(128, K, lane_major)  # a tile has at most 128 rows
    blocks = sf_view[torch.from_numpy(vs).to(sf_view.device)].cpu().numpy()
    i = rows - firsts[vs]
    return blocks[np.arange(rows.size)[:, None], idx[i]]


def sample_tokens(T, n=6):
    if T <= 48:
        return np.arange(T)
    rng = np.random.default_rng(T)
    return np.unique(np.concatenate([[0, T - 1], rng.choice(T, n - 2, replace=False)]))


def spread_tokens(T, n):
    """n tokens spread over [0, T): both ends, an even stride and random offsets
    (so they fall into many tiles of many experts)."""
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(T + n)
    base = np.linspace(0, T - 1, n).astype(np.int64)
    jit = rng.integers(-(T // n) // 2, (T // n) // 2 + 1, n)
    return np.unique(np.clip(np.concatenate([[0, T - 1], base + jit]), 0, T - 1))


# Intermediate codes that may differ from the oracle's (fp32 tensor-core sums
# against fp64 sums crossing an E4M3 rounding boundary), per activation.
# Measured on GB300: 0 % on every SwiGLU workload but the skewed one
# (0.00036 %); 0.0061 % for SiTU at the decode workload (the hardware tanh
# approximation, relative error about 2^-11).
ACT_DIFF_FRACTION = {0: 1e-3, 1: 1e-3, 2: 1e-3}


def e4m3_step(v, scale_code):
    """One E4M3 step at magnitude |v| in a block with E8M0 scale code
    `scale_code` (normal binades: 3 mantissa bits; below 2^-6 the subnormal
    step 2^-9), in absolute units."""
    s = np.exp2(scale_code.astype(np.float64) - 127)
    u = np.abs(v) / s
    e = np.floor(np.log2(np.maximum(u, 2.0 ** -6)))
    return np.exp2(e - 3) * s


def check_intermediate(ga_codes, ga_sf, oa_codes, oa_sf):
    """Decoded GPU vs oracle intermediate of one row: (#elements, #differing),
    asserting every difference is within one step (see the module header)."""
    g_sf = np.repeat(ga_sf, 32)
    o_sf = np.repeat(oa_sf, 32)
    ga = E4M3_VALUES[ga_codes] * np.exp2(g_sf.astype(np.float64) - 127)
    oa = E4M3_VALUES[oa_codes] * np.exp2(o_sf.astype(np.float64) - 127)
    d = ga != oa
    if d.any():
        mag = np.maximum(np.abs(ga[d]), np.abs(oa[d]))
        step = np.maximum(e4m3_step(mag, g_sf[d]), e4m3_step(mag, o_sf[d]))
        bad = np.abs(ga[d] - oa[d]) > step
        assert not bad.any(), (ga[d][bad][:4], oa[d][bad][:4], step[bad][:4])
    return ga.size, int(d.sum())


def out_excess(got, ref, kp):
    """Per element, how far |got - ref| exceeds the bf16 roundings on the path:
    at 128-row tiles each of the token's k' FC2 rows is rounded to bf16, and
    the output once more, each within half a bf16 step (2^-9 relative).  The
    layer's absolute bar (2e-2) applies to what is left; at the pages'
    shapes the outputs are small enough that this changes nothing, at wider
    layers (|out| of several units, a bf16 step of 0.03 and more) it keeps
    the bar about the arithmetic rather than the output's scale."""
    return np.abs(got - ref) - (kp + 1) * 2.0 ** -9 * np.abs(ref)


def check_layer(cfg, tokens=None, y_rows=True, scaled_abs=False):
    shape, ws, out, ids, w, status = run_layer(cfg)
    assert status == (0, 0), status
    orc = OracleCase(cfg)
    # routing: ids bit-exact, weights to fp32 accuracy
    np.testing.assert_array_equal(ids.cpu().numpy(), orc.ids)
    wg = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(wg - orc.w) <= 4e-6 * np.abs(orc.w) + 1e-7), np.max(np.abs(wg - orc.w))
    # sort: bit-exact
    v = moe.moe_get_views(shape, ws)
    s = orc.sort
    hdr = v["header"].cpu().numpy()
    R = int(s["offsets"][-1])
    assert hdr[0] == R and hdr[1] == s["num_v"]
    np.testing.assert_array_equal(v["expert_counts"].cpu().numpy(), s["counts"])
    np.testing.assert_array_equal(v["expert_offsets"].cpu().numpy(), s["offsets"])
    np.testing.assert_array_equal(v["c_map"].cpu().numpy()[:cfg.T * cfg.kp], s["c_map"])
    np.testing.assert_array_equal(v["a_map"].cpu().numpy()[:R], s["a_map"])
    vinfo = v["vinfo"].cpu().numpy()
    np.testing.assert_array_equal(vinfo[:s["num_v"]], s["vinfo"])
    # forward on the checked tokens
    toks = sample_tokens(cfg.T) if tokens is None else tokens
    ref = orc.forward(toks, want_y=y_rows)
    token_order = bool(v["x_token_order"])
    num_v = s["num_v"]
    # the expert rows of the checked tokens' slots, gathered on the device
    slots = [(k, j, int(s["c_map"][t * cfg.kp + j])) for k, t in enumerate(toks) for j in range(cfg.kp)
             if s["c_map"][t * cfg.kp + j] >= 0]
    rows = np.array([r for _, _, r in slots], np.int64)
    rows_t = torch.from_numpy(rows).cuda()
    act = v["act"][rows_t].cpu().numpy() if rows.size else None
    asf = tile_scales_of_rows(v["act_sf"], vinfo, num_v, cfg.inter, rows) if rows.size else None
    y = v["y"][rows_t].float().cpu().numpy() if (y_rows and rows.size) else None
    if token_order:  # x -> MXFP8 in token order: bit-exact
        tt = torch.from_numpy(np.asarray(toks, np.int64)).cuda()
        np.testing.assert_array_equal(v["xq"][tt].cpu().numpy(), ref["xq"])
        np.testing.assert_array_equal(v["xq_sf"][tt].cpu().numpy(), ref["xq_sf"])
    elif rows.size:  # x -> MXFP8 in expert-row order: bit-exact
        ks = np.array([k for k, _, _ in slots])
        np.testing.assert_array_equal(v["xq"][rows_t].cpu().numpy(), ref["xq"][ks])
        np.testing.assert_array_equal(tile_scales_of_rows(v["xq_sf"], vinfo, num_v, cfg.hidden, rows, True),
                                      ref["xq_sf"][ks])
    n_act, n_diff, y_worst, n_y = 0, 0, 0.0, 0
    for m, (k, j, row) in enumerate(slots):
        # intermediate: decoded values, mostly identical, else one step apart
        na, nd = check_intermediate(act[m], asf[m], ref["act"][k, j], ref["act_sf"][k, j])
        n_act += na
        n_diff += nd
        # the FC2 row of this slot (already times the routing weight), where
        # FC2's input equals the oracle's (the output bar covers the others)
        if y_rows and nd == 0:
            e = rel_l2(y[m], ref["y_slot"][k, j])
            y_worst = max(y_worst, e)
            n_y += 1
            assert e <= 1e-2, (toks[k], j, e)
    frac = n_diff / max(n_act, 1)
    got = bf16_to_f64(bf16_bits(out)[toks])
    err, mab = rel_l2(got, ref["out_f64"]), float(np.max(np.abs(got - ref["out_f64"])))
    if scaled_abs:
        mab = float(np.max(out_excess(got, ref["out_f64"], cfg.kp)))
    print("PARITY %s tokens=%d act_diff=%d/%d (%.3g%%) fc2_rows=%d worst_row_rel_l2=%.3g out_rel_l2=%.3g "
          "%s=%.3g" % (_cid(cfg), len(toks), n_diff, n_act, 100 * frac, n_y, y_worst, err,
                       "out_max_excess" if scaled_abs else "out_max_abs", mab))
    assert n_diff <= ACT_DIFF_FRACTION[cfg.activation] * max(n_act, 1), (n_diff, n_act)
    assert err <= 1e-2
    assert mab <= 2e-2
    return out


@pytest.mark.parametrize("cfg", GRID, ids=_cid)
def test_layer_grid_vs_oracle(cfg):
    check_layer(cfg)


# The decode verification points of the shape-template page ("correctness":
# T in {1, 7, 48, 96, 256} x BlockN in {16, 32}) on the decode layer's own
# shape: 896 experts, top-16, H 3584, I 384.  Every token is checked.
SWEEP = [synth.CONFIGS["decode_t32"].replace(T=T, block_n=B) for T in (1, 7, 48, 96, 256) for B in (16, 32)]


@pytest.mark.parametrize("cfg", SWEEP, ids=_cid)
def test_decode_shape_sweep_vs_oracle(cfg):
    check_layer(cfg, tokens=np.arange(cfg.T))


# Longer decode batches on the same shape: at T 512 the one-CTA token-bitmask
# sort runs with its largest tables (896 experts, k' 16 and 17: 180 and 186 KB
# of shared memory); past 512 tokens the general sort and the x quantiser's
# own launch.  The sorted maps are checked in full, the forward on 32 tokens
# spread over the batch.
LONG_DECODE = [synth.CONFIGS["decode_t32"].replace(T=512), synth.CONFIGS["skewed_shared_t256"].replace(T=512),
               synth.CONFIGS["decode_t32"].replace(T=600)]


@pytest.mark.parametrize("cfg", LONG_DECODE, ids=_cid)
def test_decode_long_batches_vs_oracle(cfg):
    check_layer(cfg, tokens=spread_tokens(cfg.T, 32))


# Every token on the same experts: a Zipf popularity so steep (s = 30, logit
# gaps of 20 and more between neighbouring ids against N(0, 1) noise) that
# each token's top-k is experts 0 .. k-1 in that order.  Each of them holds all
# T rows, cut into many virtual experts (tiles) of one expert: the most skewed
# routing the method meets.  A slice that holds none of those experts gets no
# routed row at all: its output is the shared expert's alone, or exactly zero.
HOT = [
    SMALL.replace(T=64, block_n=16, zipf_s=30.0),  # fused route + sort: 4 virtual experts per expert
    SMALL.replace(T=300, block_n=32, num_shared=1, zipf_s=30.0),  # route launch + one-CTA token sort
    SMALL.replace(T=600, block_n=32, zipf_s=30.0),  # general sort and the x quantiser's own launch
    SMALL.replace(T=1000, block_n=128, num_shared=1, zipf_s=30.0),  # 128-row tiles: 8 per expert
    SMALL.replace(T=200, block_n=32, E_local=32, expert_offset=32, zipf_s=30.0),  # no row at all
    SMALL.replace(T=200, block_n=128, E_local=32, expert_offset=32, num_shared=1, zipf_s=30.0),  # shared rows only
]


@pytest.mark.parametrize("cfg", HOT, ids=_cid)
def test_every_token_on_the_same_experts_vs_oracle(cfg):
    orc = OracleCase(cfg)
    np.testing.assert_array_equal(orc.ids[:, :cfg.top_k], np.tile(np.arange(cfg.top_k), (cfg.T, 1)))
    local = [e for e in range(cfg.top_k) if cfg.expert_offset <= e < cfg.expert_offset + cfg.E_local]
    counts = orc.sort["counts"]
    assert sorted(counts[counts > 0].tolist()) == [cfg.T] * (len(local) + cfg.num_shared)
    out = check_layer(cfg, tokens=spread_tokens(cfg.T, 24))
    if not local and not cfg.num_shared:
        assert not bf16_bits(out).any()  # no routed row: the output is +0 everywhere


# The largest routing shape the library takes: 1024 experts in all (1023 in the
# local slice plus the shared one fill the 1024 local slots), top-32 plus the
# shared expert (k' 33, the fused route + sort's limit), through the fused,
# one-CTA and ballot sorts and the 128-row tiling.
MAXR = SMALL.replace(E_global=1024, E_local=1023, expert_offset=1, top_k=32, num_shared=1, hidden=512, inter=128)
MAX_ROUTING = [MAXR.replace(T=16, block_n=16), MAXR.replace(T=200, block_n=32), MAXR.replace(T=600, block_n=32),
               MAXR.replace(T=300, block_n=128)]


@pytest.mark.parametrize("cfg", MAX_ROUTING, ids=_cid)
def test_largest_routing_shape_vs_oracle(cfg):
    assert moe.moe_is_supported(shape_of(cfg))
    assert not moe.moe_is_supported(shape_of(cfg.replace(E_local=1024, expert_offset=0)))  # 1025 local slots
    check_layer(cfg, tokens=spread_tokens(cfg.T, 16))


@pytest.mark.parametrize("cfg", [SMALL.replace(T=16, block_n=16, E_global=896, E_local=896, top_k=16),
                                 SMALL.replace(T=100, block_n=32, E_global=896, E_local=896, top_k=16, num_shared=1),
                                 SMALL.replace(T=200, block_n=128, top_k=8)], ids=_cid)
def test_all_logits_equal_vs_oracle(cfg):
    # every logit of every token equal (zero): the routing's heaviest tie
    # (all experts candidates, the selection's fallback over all entries);
    # ties go to the lower id, so each token takes experts 0 .. k-1 with
    # weight 1/k, and the layer must still match the oracle
    shape = shape_of(cfg)
    x, logits, sl = device_inputs(cfg)
    logits = torch.zeros_like(logits)
    ws = moe.workspace(shape)
    out, ids, w = moe.moe_layer(shape, logits, sl, x, _weights(cfg), ws)
    torch.cuda.synchronize()
    assert moe.moe_get_status(ws) == (0, 0)
    orc = OracleCase(cfg, logits=np.zeros((cfg.T, cfg.E_global), np.float32))
    np.testing.assert_array_equal(orc.ids[:, :cfg.top_k], np.tile(np.arange(cfg.top_k), (cfg.T, 1)))
    np.testing.assert_array_equal(ids.cpu().numpy(), orc.ids)
    wg = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(wg - orc.w) <= 4e-6 * np.abs(orc.w) + 1e-7)
    assert np.allclose(wg[:, :cfg.top_k], 1.0 / cfg.top_k, rtol=1e-6)
    toks = spread_tokens(cfg.T, 8)
    ref = orc.forward(toks)["out_f64"]
    got = bf16_to_f64(bf16_bits(out)[toks])
    assert rel_l2(got, ref) <= 1e-2 and float(np.max(np.abs(got - ref))) <= 2e-2


# Wide layers: hidden 7168 and inter 2048 (14 / 16 K chunks per FC2 / FC1
# item, 28 FC2 weight blocks and 16 FC1 blocks per expert), on both tilings
# and both GEMM2 paths (nothing in the kernels is sized by H or I).
WIDE = SMALL.replace(E_global=8, E_local=8, top_k=2, num_shared=1, hidden=7168, inter=2048)


@pytest.mark.parametrize("cfg", [WIDE.replace(T=40, block_n=32), WIDE.replace(T=300, block_n=128)], ids=_cid)
def test_wide_layer_vs_oracle(cfg):
    # outputs of several units here: the absolute bar applies beyond the bf16
    # roundings of the path (out_excess)
    check_layer(cfg, tokens=spread_tokens(cfg.T, 8), scaled_abs=True)
    shape = shape_of(cfg)
    x, logits, sl = device_inputs(cfg)
    ws = moe.workspace(shape)
    moe.moe_set_gemm2_path(moe.GEMM2_DENSE)
    try:
        out, _, _ = moe.moe_layer(shape, logits, sl, x, _weights(cfg), ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_gemm2_path(moe.GEMM2_AUTO)
    assert moe.moe_get_status(ws) == (0, 0)
    toks = spread_tokens(cfg.T, 8)
    ref = OracleCase(cfg).forward(toks)["out_f64"]
    got = bf16_to_f64(bf16_bits(out)[toks])
    assert rel_l2(got, ref) <= 1e-2 and float(np.max(out_excess(got, ref, cfg.kp))) <= 2e-2


@pytest.mark.parametrize("cfg", [SMALL.replace(T=37, block_n=32), SMALL.replace(T=600, block_n=16, num_shared=1),
                                 SMALL.replace(T=300, block_n=128)], ids=_cid)
def test_workspace_sized_for_a_larger_batch(cfg):
    # A workspace carved for max_T 4096, first filled by a 4096-token call, then
    # called with T tokens: the ids, weights and output equal those of a call on
    # a workspace carved for exactly T -- bit for bit on the split path, within
    # the dense path's run-to-run bound (its reductions run in no fixed order;
    # dense_repeat_bound).  Nothing a call reads may come from a region sized
    # by max_T but written only by an earlier, larger call.
    wts = _weights(cfg)
    x, logits, sl = device_inputs(cfg)
    xb, lb, sb = device_inputs(cfg, T=4096)
    exact, big = shape_of(cfg), shape_of(cfg)
    big.max_T = 4096
    full = shape_of(cfg, T=4096)
    for path in (moe.GEMM2_SPLIT, moe.GEMM2_DENSE):
        moe.moe_set_gemm2_path(path)
        try:
            ws_e, ws_b = moe.workspace(exact), moe.workspace(big)
            a = moe.moe_layer(exact, logits, sl, x, wts, ws_e)
            moe.moe_layer(full, lb, sb, xb, wts, ws_b)
            b = moe.moe_layer(big, logits, sl, x, wts, ws_b)
            torch.cuda.synchronize()
        finally:
            moe.moe_set_gemm2_path(moe.GEMM2_AUTO)
        assert moe.moe_get_status(ws_e) == (0, 0) and moe.moe_get_status(ws_b) == (0, 0)
        assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
        if path == moe.GEMM2_SPLIT:
            assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
            slack = dense_repeat_bound(exact, ws_e, cfg.T)  # the split rows of ws_e, for the dense check
        else:
            fa, fb = a[0].double().cpu().numpy(), b[0].double().cpu().numpy()
            assert within_dense_repeat(fa, fb, slack)


@pytest.mark.parametrize("cfg", FULL, ids=_cid)
def test_layer_full_size_vs_oracle(cfg):
    # every token of the decode workloads; 64 tokens spread over the prefill
    # (and so over many tiles of every expert)
    check_layer(cfg, tokens=np.arange(cfg.T) if cfg.T <= 256 else spread_tokens(cfg.T, 64))


@pytest.mark.parametrize("act,params", [(1, (7.0, 0.0)), (2, (4.0, 25.0))])
def test_decode_layer_activation_variants_vs_oracle(act, params):
    # the decode layer with the clamped SwiGLU at the usual limit 7 and SiTU
    # with the constants the shape-templates page fixes (beta 4, lb 25)
    check_layer(synth.CONFIGS["decode_t32"].replace(activation=act, act_params=params), tokens=sample_tokens(32, 4))


def test_weight_quantiser_bit_exact():
    cfg = SMALL.replace(E_local=4, E_global=4, hidden=512, inter=128)
    _, (c1, s1, _, _) = device_weights(cfg, keep_rowmajor=True)
    f1 = synth.w1_host(cfg, cfg.global_ids)
    for e in range(4):
        c, s = oracle.quantize_mxfp4(f1[e])
        np.testing.assert_array_equal(c1[e].cpu().numpy(), c)
        np.testing.assert_array_equal(s1[e].cpu().numpy(), s)
    # edge values: zeros, exact ties, saturation, tiny and huge blocks
    rng = np.random.default_rng(3)
    w = (rng.integers(-14, 15, (256, 64)) * 0.25 * 2.0 ** rng.integers(-8, 8, (256, 1))).astype(np.float32)
    w[0] = 0
    w[1, :32] = -0.0
    w[2] = rng.normal(0, 1e-30, 64)
    w[3] = rng.normal(0, 1e30, 64)
    w[4, 5] = 7.0
    w[4, :5] = 4.0
    c, s = moe.moe_quantize_mxfp4(torch.from_numpy(w).cuda())
    oc, os_ = oracle.quantize_mxfp4(w)
    np.testing.assert_array_equal(c.cpu().numpy(), oc)
    np.testing.assert_array_equal(s.cpu().numpy(), os_)


@pytest.mark.parametrize("pair", [False, True])
def test_pack_weights_layout(pair):
    E, N, K = 2, 512, 384
    codes = torch.randint(0, 255, (E, N, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.randint(0, 255, (E, N, K // 32), dtype=torch.uint8, device="cuda")
    pc, ps = moe.moe_pack_weights(codes, scales, pair)
    pc, ps = pc.cpu().numpy(), ps.cpu().numpy()
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    NB, KC = N // 256, K // 128
    for e in range(E):
        for b in range(NB):
            rows = (list(range(b * 128, b * 128 + 128)) + list(range(N // 2 + b * 128, N // 2 + b * 128 + 128))
                    if pair else list(range(b * 256, b * 256 + 256)))
            for kc in range(KC):
                tile = (e * NB + b) * KC + kc
                tc = pc[tile * 256 * 64:(tile + 1) * 256 * 64].reshape(256, 64)
                np.testing.assert_array_equal(tc, c[e, rows, kc * 64:(kc + 1) * 64])
                ts = ps[tile * 1024:(tile + 1) * 1024]
                for rr, row in enumerate(rows):
                    g, r = rr // 128, rr % 128
                    for j in range(4):
                        assert ts[g * 512 + (r % 32) * 16 + (r // 32) * 4 + j] == s[e, row, kc * 4 + j]


def test_synth_generators_agree():
    for stream in (1, 4):
        h = synth.normal_q16_host(9, stream, 12345, 4096)
        d = synth.normal_q16_device(9, stream, 12345, 4096).cpu().numpy()
        np.testing.assert_array_equal(h, d)
    cfg = synth.CONFIGS["skewed_shared_t256"].replace(T=8)
    np.testing.assert_array_equal(synth.logits_host(cfg), synth.logits_device(cfg).cpu().numpy())
    np.testing.assert_array_equal(synth.x_host(cfg), bf16_bits(synth.x_device(cfg)))


def _tie_logits(T, Eg, seed, coarse):
    """Logits on a 0.5 grid (coarse: heavy ties at the top, the selection's
    fallback path) or plain normal draws (its candidate path)."""
    rng = np.random.default_rng(seed)
    lg = rng.normal(0, 1, (T, Eg))
    if coarse:
        lg = np.round(lg * 2) / 2
    return lg.astype(np.float32)


def _check_sort_views(shape, ws, ref, T, kp):
    v = moe.moe_get_views(shape, ws)
    R = int(ref["offsets"][-1])
    hdr = v["header"].cpu().numpy()
    assert hdr[0] == R and hdr[1] == ref["num_v"] and hdr[3] == 0
    np.testing.assert_array_equal(v["expert_counts"].cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(v["expert_offsets"].cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(v["c_map"].cpu().numpy()[:T * kp], ref["c_map"])
    np.testing.assert_array_equal(v["a_map"].cpu().numpy()[:R], ref["a_map"])
    np.testing.assert_array_equal(v["vinfo"].cpu().numpy()[:ref["num_v"]], ref["vinfo"])


@pytest.mark.parametrize("Eg,k,coarse", [(8, 2, True), (33, 5, False), (896, 16, True), (896, 16, False),
                                         (1024, 32, True), (1024, 32, False), (640, 1, True)])
def test_route_kernel_exact_with_and_without_ties(Eg, k, coarse):
    T = 300
    lg = _tie_logits(T, Eg, Eg + k, coarse)
    shape = moe.MoeShape(T=T, max_T=T, E_global=Eg, E_local=Eg, expert_offset=0, top_k=k, num_shared=0,
                         hidden=512, inter=128, block_n=32)
    ids, w = moe.moe_route(shape, torch.from_numpy(lg).cuda())
    torch.cuda.synchronize()
    oids, ow = oracle.route(lg, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), oids)
    wg = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(wg - ow) <= 4e-6 * np.abs(ow) + 1e-7)


@pytest.mark.parametrize("T,coarse,S", [(32, True, 0), (64, False, 0), (48, True, 1), (7, False, 1), (100, True, 1),
                                         (128, False, 0), (128, True, 1)])
def test_fused_and_split_route_sort_agree_with_oracle(T, coarse, S):
    # moe_layer ranks its own routing with token bitmasks: in the fused route
    # + sort kernel up to 64 tokens, in a one-CTA sort after the route launch
    # up to 512; moe_route + moe_sort run the general kernels.  Both must give
    # the oracle's maps.
    cfg = SMALL.replace(T=T, top_k=16, num_shared=S, E_local=64, block_n=32)
    shape = shape_of(cfg)
    assert shape.T <= 512
    lg = _tie_logits(T, cfg.E_global, T + S, coarse)
    x, _, sl = device_inputs(cfg)
    oids, ow = oracle.route(lg, cfg.top_k, S, synth.shared_logit_host(cfg) if S else None, cfg.shared_scale)
    ref = oracle.sort(oids, cfg.E_global, cfg.E_local, cfg.expert_offset, S, cfg.block_n)
    lgd = torch.from_numpy(lg).cuda()
    ws = moe.workspace(shape)
    _, ids, w = moe.moe_layer(shape, lgd, sl, x, _weights(cfg), ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), oids)
    assert np.all(np.abs(w.cpu().numpy() - ow) <= 4e-6 * np.abs(ow) + 1e-7)
    _check_sort_views(shape, ws, ref, T, shape.kp)
    ws2 = moe.workspace(shape)
    ids2, _ = moe.moe_route(shape, lgd, sl)
    moe.moe_sort(shape, ids2, ws2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids2.cpu().numpy(), oids)
    _check_sort_views(shape, ws2, ref, T, shape.kp)


@pytest.fixture
def split_path():
    """Bit-reproducibility checks run on the split GEMM2 path (the dense path
    reduces in no fixed order; see test_gpu_gemm2_gate.py)."""
    moe.moe_set_gemm2_path(moe.GEMM2_SPLIT)
    yield
    moe.moe_set_gemm2_path(moe.GEMM2_AUTO)


def test_deterministic_and_status_ok(split_path):
    cfg = GRID[3]
    _, ws, out1, _, _, st = run_layer(cfg)
    _, ws2, out2, _, _, st2 = run_layer(cfg)
    assert st == (0, 0) and st2 == (0, 0)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_expert_parallel_slices_sum_to_full():
    full_cfg = SMALL.replace(T=64, block_n=16)
    _, _, full, _, _, st = run_layer(full_cfg)
    assert st == (0, 0)
    acc = torch.zeros_like(full, dtype=torch.float32)
    for off in (0, 32):
        c = full_cfg.replace(E_local=32, expert_offset=off)
        _, _, part, _, _, st = run_layer(c)
        assert st == (0, 0)
        acc += part.float()
    # each slice rounds to bf16 on its own: allow two bf16 roundings
    assert rel_l2(acc.cpu().numpy(), full.float().cpu().numpy()) <= 1e-2
    assert torch.max(torch.abs(acc - full.float())).item() <= 2e-2


def test_zero_tokens_and_single_token():
    cfg = SMALL.replace(T=1, block_n=32)
    check_layer(cfg)
    shape = shape_of(cfg, 0)
    shape.max_T = 4
    wts = _weights(cfg)
    ws = moe.workspace(shape)
    x = torch.empty((0, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    lg = torch.empty((0, cfg.E_global), dtype=torch.float32, device="cuda")
    out, ids, w = moe.moe_layer(shape, lg, None, x, wts, ws)
    torch.cuda.synchronize()
    assert out.shape == (0, cfg.hidden)


def test_graph_capture_replays_the_chain(split_path):
    cfg = GRID[2]
    shape = shape_of(cfg)
    wts = _weights(cfg)
    x, logits, sl = device_inputs(cfg)
    ws = moe.workspace(shape)
    ids = torch.empty((shape.T, shape.kp), dtype=torch.int32, device="cuda")
    w = torch.empty((shape.T, shape.kp), dtype=torch.float32, device="cuda")
    out = torch.empty((shape.T, shape.hidden), dtype=torch.bfloat16, device="cuda")
    ref, _, _ = moe.moe_layer(shape, logits, sl, x, wts, ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            moe.moe_layer(shape, logits, sl, x, wts, ws, ids, w, out)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert moe.moe_get_status(ws) == (0, 0)


@pytest.mark.parametrize("cfg", [GRID[2], GRID[6], GRID[9], SMALL.replace(T=5, block_n=128, num_shared=1)],
                         ids=_cid)
def test_host_buffer_entry_point_matches_device_path(split_path, cfg):
    # 128-row tilings take the pipelined form (copies in token chunks on a
    # second stream, overlapped with the gather and the combine; at T 5 most
    # chunks are empty); two calls in a row on one workspace reuse its staging
    shape = shape_of(cfg)
    wts = _weights(cfg)
    x, logits, sl = device_inputs(cfg)
    ws = moe.workspace(shape)
    ref, _, _ = moe.moe_layer(shape, logits, sl, x, wts, ws)
    xh, lh = x.cpu().pin_memory(), logits.cpu().pin_memory()
    sh = sl.cpu().pin_memory() if sl is not None else None
    ws2 = moe.workspace(shape)
    for _ in range(2):
        oh = torch.full((shape.T, shape.hidden), float("nan"), dtype=torch.bfloat16).pin_memory()
        moe.moe_layer_host(shape, lh, sh, xh, wts, ws2, oh)
        torch.cuda.synchronize()
        assert moe.moe_get_status(ws2) == (0, 0)
        assert torch.equal(oh.view(torch.int16), ref.cpu().view(torch.int16))


@pytest.mark.parametrize("cfg", [GRID[5], GRID[6]], ids=_cid)
def test_layers_on_two_streams_run_independently(split_path, cfg):
    # moe_layer calls alternating over two streams, each with its own
    # workspace and inputs, issued without host synchronisation, so that their
    # launches can overlap on the GPU: the chain keeps no state outside its
    # workspace, and each output equals its own call's alone, bit for bit
    shape = shape_of(cfg)
    wts = _weights(cfg)
    x, logits, sl = device_inputs(cfg)
    flip = lambda t: t.flip(0).contiguous() if t is not None else None  # noqa: E731
    inputs = [(x, logits, sl), (flip(x), flip(logits), flip(sl))]
    ws0 = moe.workspace(shape)
    refs = []
    for xx, lg, s_ in inputs:
        out, ids, w = moe.moe_layer(shape, lg, s_, xx, wts, ws0)
        refs.append((out.clone(), ids.clone(), w.clone()))
    torch.cuda.synchronize()
    wss = [moe.workspace(shape), moe.workspace(shape)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    results = []
    for i in range(6):
        xx, lg, s_ = inputs[i % 2]
        with torch.cuda.stream(streams[i % 2]):
            results.append(moe.moe_layer(shape, lg, s_, xx, wts, wss[i % 2]))
    torch.cuda.synchronize()
    for i, (out, ids, w) in enumerate(results):
        r_out, r_ids, r_w = refs[i % 2]
        assert torch.equal(ids, r_ids), i
        assert torch.equal(w, r_w), i
        assert torch.equal(out.view(torch.int16), r_out.view(torch.int16)), i
    for w_ in wss:
        assert moe.moe_get_status(w_) == (0, 0)


def test_host_buffer_calls_on_two_streams(split_path):
    # consecutive moe_layer_host calls alternating over two caller streams,
    # each stream with its own workspace, different inputs per stream and no
    # host synchronisation between calls: one call's output copies overlap
    # the next call's input copies and compute, and each output must still be
    # its own call's, bit for bit
    cfg = GRID[9]
    shape = shape_of(cfg)
    wts = _weights(cfg)
    x, logits, sl = device_inputs(cfg)
    flip = lambda t: t.flip(0).contiguous() if t is not None else None  # noqa: E731
    inputs = [(x, logits, sl), (flip(x), flip(logits), flip(sl))]
    ws0 = moe.workspace(shape)
    refs = [moe.moe_layer(shape, lg, s_, xx, wts, ws0)[0].cpu() for xx, lg, s_ in inputs]
    assert not torch.equal(refs[0], refs[1])
    pin = lambda t: t.cpu().pin_memory() if t is not None else None  # noqa: E731
    host = [(pin(xx), pin(lg), pin(s_)) for xx, lg, s_ in inputs]
    wss = [moe.workspace(shape), moe.workspace(shape)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.full((shape.T, shape.hidden), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in range(6)]
    torch.cuda.synchronize()
    for i, oh in enumerate(outs):
        xh, lh, sh = host[i % 2]
        with torch.cuda.stream(streams[i % 2]):
            moe.moe_layer_host(shape, lh, sh, xh, wts, wss[i % 2], oh)
    torch.cuda.synchronize()
    for i, oh in enumerate(outs):
        assert torch.equal(oh.view(torch.int16), refs[i % 2].view(torch.int16)), i
    for w in wss:
        assert moe.moe_get_status(w) == (0, 0)


# ----------------------------------------------------------------- edge values
def _e4m3_midpoints(rng, n):
    """Values half-way between two adjacent positive normal E4M3 codes (exact
    in bf16: one bit more than E4M3's three mantissa bits)."""
    codes = rng.integers(0x08, 0x7D, n)
    return (E4M3_VALUES[codes] + E4M3_VALUES[codes + 1]) / 2


def edge_x_bits(T, H, seed):
    """bf16 bits [T, H]: normal draws, with one MX block of every row replaced
    by an edge case (cycling over the rows): all +0, all -0, bf16 subnormals,
    a block holding the bf16 maximum, an amax exactly on a power of two, E4M3
    ties (block scale 2^0), amaxes in (448, 512) that saturate, and tiny
    values that underflow to a signed zero next to a large amax.  Row 0 is
    zero throughout."""
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.normal(0, 1, (T, H)).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16).copy()

    def to_bits(v):
        return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    for t in range(T):
        b = (3 * t + 1) % (H // 32)
        blk = slice(32 * b, 32 * b + 32)
        kind = t % 8
        sign = rng.integers(0, 2, 32).astype(np.uint16) << 15
        if kind == 0:
            bits[t, blk] = 0
        elif kind == 1:
            bits[t, blk] = 0x8000
        elif kind == 2:
            bits[t, blk] = rng.integers(1, 128, 32).astype(np.uint16) | sign
        elif kind == 3:
            v = rng.normal(0, 1e37, 32)
            bits[t, blk] = to_bits(v)
            bits[t, 32 * b + rng.integers(0, 32)] = 0x7F7F | (int(sign[0]) & 0x8000)
        elif kind == 4:
            k = int(rng.integers(-20, 21))
            v = rng.uniform(-1, 1, 32) * 2.0 ** k
            v[rng.integers(0, 32)] = -(2.0 ** k) if sign[1] else 2.0 ** k
            bits[t, blk] = to_bits(v)
        elif kind == 5:
            v = _e4m3_midpoints(rng, 32) * np.where(sign > 0, -1, 1)
            v[0] = 256.0  # amax 256: block scale 2^0, codes are the values themselves
            bits[t, blk] = to_bits(v)
        elif kind == 6:
            v = rng.uniform(-480, 480, 32)
            v[:4] = [448.0, -456.0, 480.0, 500.0]  # 456 / 480 / 500 saturate to 448
            bits[t, blk] = to_bits(v)
        else:
            v = rng.uniform(-1e-5, 1e-5, 32)  # below half the smallest step: signed zeros
            v[7] = 1024.0
            bits[t, blk] = to_bits(v)
    bits[0] = 0
    return bits


@pytest.mark.parametrize("T,block_n,path", [(16, 32, "fused route+sort"), (128, 32, "route launch"),
                                            (600, 16, "quant_x launch"), (64, 128, "token-major gather")])
def test_x_quantiser_edge_values_all_paths(T, block_n, path):
    # x -> MXFP8 is computed by four launches depending on the tiling and
    # batch: inside the fused route + sort (decode tilings, T <= 64), in the
    # route launch (decode tilings, T <= 512), by its own launch (decode
    # tilings, larger batches) and by the token-major gather into expert rows
    # (128-row tiles).  All must equal the oracle's
    # quantiser bit for bit on edge values.
    cfg = SMALL.replace(T=T, block_n=block_n, top_k=4)
    shape = shape_of(cfg)
    if block_n < 128:  # 128-row tiles quantise x in the gather even when route and sort are fused
        expect = "fused route+sort" if shape.T <= 64 else ("route launch" if shape.T <= 512 else "quant_x launch")
        assert path == expect
    bits = edge_x_bits(T, cfg.hidden, T + block_n)
    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    _, logits, sl = device_inputs(cfg)
    ws = moe.workspace(shape)
    moe.moe_layer(shape, logits, sl, x, _weights(cfg), ws)
    torch.cuda.synchronize()
    assert moe.moe_get_status(ws) == (0, 0)
    oq, osf = oracle.quantize_mxfp8_bf16(bits)
    v = moe.moe_get_views(shape, ws)
    if v["x_token_order"]:
        np.testing.assert_array_equal(v["xq"][:T].cpu().numpy(), oq)
        np.testing.assert_array_equal(v["xq_sf"][:T].cpu().numpy(), osf)
    else:
        R = int(v["header"][0].item())
        tok = v["a_map"][:R].cpu().numpy() // shape.kp
        vinfo = v["vinfo"].cpu().numpy()
        np.testing.assert_array_equal(v["xq"][:R].cpu().numpy(), oq[tok])
        np.testing.assert_array_equal(
            tile_scales_of_rows(v["xq_sf"], vinfo, int(v["header"][1].item()), cfg.hidden, np.arange(R), True),
            osf[tok])
    # the cases are really there: zero, negative-zero and saturated codes
    assert (oq == 0x80).any() and (oq == 0x7E).any() and (osf == 0).any()


@pytest.mark.parametrize("T,block_n", [(100, 32), (100, 128), (3000, 16), (3000, 128)])
def test_sort_masked_out_of_slice_and_duplicate_ids(T, block_n):
    # moe_sort on ids a caller hands in: masked (-1 and other negatives), ids
    # of other ranks' slices, ids past the shared expert, the shared id, and a
    # token naming one expert twice.  T * k' = 700 takes the one-CTA sort,
    # 21000 the count / scan / rank kernels.  Bit-exact against the oracle
    # ("... MXFP4 decode MoE ... shape templates", section 5: ids outside the
    # local slice get no row).
    Eg, El, off, S, k = 256, 128, 64, 1, 6
    shape = moe.MoeShape(T=T, max_T=T, E_global=Eg, E_local=El, expert_offset=off, top_k=k, num_shared=S,
                         hidden=1024, inter=256, block_n=block_n)
    rng = np.random.default_rng(T + block_n)
    ids = rng.integers(-3, 300, (T, k + S)).astype(np.int32)
    ids[:, k] = Eg  # the shared slot
    ids[::7, 1] = ids[::7, 0]  # duplicates within a token
    ids[::5, 2] = -1
    ids[1, :] = -1  # a token with no row at all
    ws = moe.workspace(shape)
    moe.moe_sort(shape, torch.from_numpy(ids).cuda(), ws)
    torch.cuda.synchronize()
    ref = oracle.sort(ids, Eg, El, off, S, block_n)
    _check_sort_views(shape, ws, ref, T, shape.kp)
    assert (ref["c_map"] < 0).sum() > T  # many slots without a row
