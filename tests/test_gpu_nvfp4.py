"""The NVFP4 variant through the C ABI (marked gpu): "[SGLang] CUTLASS MoE",
section 6 -- E2M1 activations and weights in blocks of 16 with E4M3 scales and
fp32 global scales, on tcgen05 kind::mxf4nvf4 tensor cores, 128-row tiles.

Bars as in test_gpu_parity.py: the weight quantiser (global scales, codes,
block scales) and the packed layouts bit-exact; routing and sort bit-exact;
NVFP4(x) codes and scales bit-exact; intermediate codes at most 0.1 %
different, each within one E2M1 step at the coarser of the two block scales;
each FC2 row (split path) whose intermediate equals the oracle's within
relative L2 1e-2; output relative L2 <= 1e-2 and max-abs <= 2e-2 against the
oracle's own NVFP4 forward."""
import numpy as np
import pytest
import torch

import mxfp4_mixture_experts_02_gb300 as moe
import oracle
import synth
from moe_case import (OracleCase, bf16_bits, bf16_to_f64, device_inputs, device_weights_nvfp4, rel_l2, shape_of)

pytestmark = pytest.mark.gpu

X_GS = 448.0      # x ~ N(0, 1) within +-6: 2688 / 6
H_GS = 42.0       # the intermediate within +-64
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E4M3 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()

SMALL = synth.MoeConfig("small", 7, T=200, E_global=64, E_local=64, expert_offset=0, top_k=8, num_shared=0,
                        hidden=1024, inter=256, block_n=128)
CASES = [
    SMALL,
    SMALL.replace(T=64, E_local=32, expert_offset=32, hidden=1536, inter=384, num_shared=1),
    SMALL.replace(T=1200, E_global=8, E_local=8, top_k=2, hidden=3584, inter=128),
    SMALL.replace(T=96, activation=2, act_params=(4.0, 25.0)),
]


def _cid(c):
    return "%s-T%d-E%d+%d-S%d-H%d-I%d-A%d" % (c.name, c.T, c.E_local, c.expert_offset, c.num_shared, c.hidden,
                                               c.inter, c.activation)


def test_weight_quantiser_and_packer_bit_exact():
    cfg = SMALL.replace(E_global=4, E_local=4, hidden=512, inter=256)
    w1 = synth.w1_device(cfg, cfg.global_ids)  # [4, 2I, H]
    gs, codes, scales = moe.moe_quantize_nvfp4(w1)
    f1 = synth.w1_host(cfg, cfg.global_ids)
    for e in range(4):
        g = oracle.nvfp4_global_scale(f1[e])
        assert gs[e].item() == np.float32(g)
        c, sc = oracle.quantize_nvfp4(f1[e], g)
        np.testing.assert_array_equal(codes[e].cpu().numpy(), c)
        np.testing.assert_array_equal(scales[e].cpu().numpy(), sc)
    # edge values: a zero block, exact grid values, huge and tiny magnitudes
    rng = np.random.default_rng(5)
    w = (rng.integers(-6, 7, (1, 64, 64)) * 0.5 * 2.0 ** rng.integers(-20, 20, (1, 64, 1))).astype(np.float32)
    w[0, 0] = 0
    w[0, 1, :16] = -0.0
    w[0, 2] = rng.normal(0, 1e-30, 64)
    g, c, sc = moe.moe_quantize_nvfp4(torch.from_numpy(w).cuda())
    og = oracle.nvfp4_global_scale(w[0])
    assert g[0].item() == np.float32(og)
    oc, osc = oracle.quantize_nvfp4(w[0], og)
    np.testing.assert_array_equal(c[0].cpu().numpy(), oc)
    np.testing.assert_array_equal(sc[0].cpu().numpy(), osc)
    # packed scales: per (expert, 256-row block, 128-K chunk) 2 KiB, two 64-K halves of two 512-byte blocks
    E, N, K = 2, 512, 384
    codes = torch.randint(0, 255, (E, N, K // 2), dtype=torch.uint8, device="cuda")
    scl = torch.randint(0, 127, (E, N, K // 16), dtype=torch.uint8, device="cuda")
    for pair in (False, True):
        pc, ps = moe.moe_pack_weights_nvfp4(codes, scl, pair)
        pc, ps, cc, ss = pc.cpu().numpy(), ps.cpu().numpy(), codes.cpu().numpy(), scl.cpu().numpy()
        NB, KC = N // 256, K // 128
        for e in range(E):
            for b in range(NB):
                rows = (list(range(b * 128, b * 128 + 128)) + list(range(N // 2 + b * 128, N // 2 + b * 128 + 128))
                        if pair else list(range(b * 256, b * 256 + 256)))
                for kc in range(KC):
                    tile = (e * NB + b) * KC + kc
                    np.testing.assert_array_equal(pc[tile * 16384:(tile + 1) * 16384].reshape(256, 64),
                                                  cc[e, rows, kc * 64:(kc + 1) * 64])
                    ts = ps[tile * 2048:(tile + 1) * 2048]
                    for rr, row in enumerate(rows):
                        for kk in range(2):
                            for bb in range(4):
                                pos = kk * 1024 + (rr // 128) * 512 + (rr % 32) * 16 + ((rr % 128) // 32) * 4 + bb
                                assert ts[pos] == ss[e, row, kc * 8 + kk * 4 + bb]


def nv_scales_of_rows(ws_view, vinfo, num_v, K, rows, lane_major=False):
    """E4M3 scales [len(rows), K/16] of expert rows from the NVFP4 tile layout.
    Chunk-major (the intermediate): per virtual expert and 128-K chunk 1 KiB,
    64-K half kk at kk * 512, tile row i's cell at (i % 32) * 16 + (i / 32) * 4,
    byte = the half's block.  Lane-major (x): the same 16-byte cells ordered
    (half, lane, chunk): cell ((kk * 32 + i % 32) * (K / 128) + chunk) * 16."""
    rows = np.asarray(rows, np.int64)
    firsts = vinfo[:num_v, 1].astype(np.int64)
    vs = np.searchsorted(firsts, rows, side="right") - 1
    i = (rows - firsts[vs])[:, None]
    blk = np.arange(K // 16)[None, :]
    if lane_major:
        idx = ((((blk // 4) % 2) * 32 + i % 32) * (K // 128) + blk // 8) * 16 + (i // 32) * 4 + (blk % 4)
    else:
        idx = (blk // 8) * 1024 + ((blk // 4) % 2) * 512 + (i % 32) * 16 + (i // 32) * 4 + (blk % 4)
    tiles = ws_view[torch.from_numpy(vs).to(ws_view.device)].cpu().numpy()
    return tiles[np.arange(rows.size)[:, None], idx]


def unpack(codes):
    lo, hi = codes & 0xF, codes >> 4
    return np.stack([lo, hi], -1).reshape(codes.shape[0], -1)


def decoded(codes, sf, gs):
    return E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0) * np.repeat(E4M3[sf], 16, axis=-1) / gs


def check_layer_nvfp4(cfg, tokens, path=moe.GEMM2_SPLIT):
    shape = shape_of(cfg)
    wts, nv = device_weights_nvfp4(cfg, X_GS, H_GS)
    x, logits, sl = device_inputs(cfg)
    ws = moe.workspace(shape)
    moe.moe_set_gemm2_path(path)
    try:
        out, ids, w = moe.moe_layer_nvfp4(shape, nv, logits, sl, x, wts, ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_gemm2_path(moe.GEMM2_AUTO)
    assert moe.moe_get_status(ws) == (0, 0)
    orc = OracleCase(cfg)
    np.testing.assert_array_equal(ids.cpu().numpy(), orc.ids)
    v = moe.moe_get_views(shape, ws)
    s = orc.sort
    vinfo = v["vinfo"].cpu().numpy()
    np.testing.assert_array_equal(vinfo[:s["num_v"]], s["vinfo"])
    np.testing.assert_array_equal(v["c_map"].cpu().numpy()[:cfg.T * cfg.kp], s["c_map"])
    ref = orc.forward_nvfp4(tokens, X_GS, H_GS, want_y=True)
    H, I, nvv = cfg.hidden, cfg.inter, v["max_v"]
    base = ws.data_ptr()

    def region(t, nbytes):
        off = t.data_ptr() - base
        return ws[off:off + nbytes]

    xq = region(v["xq"], v["rows_alloc"] * H // 2).view(v["rows_alloc"], H // 2)
    xsf = region(v["xq_sf"], nvv * (H // 128) * 1024).view(nvv, (H // 128) * 1024)
    act = region(v["act"], v["rows_alloc"] * I // 2).view(v["rows_alloc"], I // 2)
    asf = region(v["act_sf"], nvv * (I // 128) * 1024).view(nvv, (I // 128) * 1024)
    slots = [(k, j, int(s["c_map"][t * cfg.kp + j])) for k, t in enumerate(tokens) for j in range(cfg.kp)
             if s["c_map"][t * cfg.kp + j] >= 0]
    rows = np.array([r for _, _, r in slots], np.int64)
    rt = torch.from_numpy(rows).cuda()
    ks = np.array([k for k, _, _ in slots])
    # x -> NVFP4 in expert-row order: bit-exact
    np.testing.assert_array_equal(unpack(xq[rt].cpu().numpy()), ref["xq"][ks])
    np.testing.assert_array_equal(nv_scales_of_rows(xsf, vinfo, s["num_v"], H, rows, True), ref["xq_sf"][ks])
    # intermediate: decoded values mostly identical, else one E2M1 step apart
    ga_c = unpack(act[rt].cpu().numpy())
    ga_s = nv_scales_of_rows(asf, vinfo, s["num_v"], I, rows)
    y = v["y"][rt].float().cpu().numpy()
    n_act = n_diff = 0
    for m, (k, j, row) in enumerate(slots):
        oc, osf = ref["act"][k, j], ref["act_sf"][k, j]
        ga, oa = decoded(ga_c[m], ga_s[m], H_GS), decoded(oc, osf, H_GS)
        d = ga != oa
        n_act += ga.size
        n_diff += int(d.sum())
        if d.any():
            mag = np.maximum(np.abs(ga[d]), np.abs(oa[d]))
            sc = np.maximum(np.repeat(E4M3[ga_s[m]], 16), np.repeat(E4M3[osf], 16))[d] / H_GS
            u = mag / sc
            step = np.where(u > 4, 2.0, np.where(u > 2, 1.0, 0.5)) * sc
            assert np.all(np.abs(ga[d] - oa[d]) <= step * (1 + 1e-9)), (row, ga[d][:4], oa[d][:4])
        # FC2 row: compared where FC2's input is the oracle's (a flipped code
        # on the 8-level E2M1 grid moves a row by a few percent; the output bar
        # covers those slots)
        if path == moe.GEMM2_SPLIT and not d.any():
            assert rel_l2(y[m], ref["y_slot"][k, j]) <= 1e-2
    got = bf16_to_f64(bf16_bits(out)[tokens])
    err, mab = rel_l2(got, ref["out_f64"]), float(np.max(np.abs(got - ref["out_f64"])))
    print("NVFP4 %s path=%d tokens=%d act_diff=%d/%d out_rel_l2=%.3g out_max_abs=%.3g" % (
        _cid(cfg), path, len(tokens), n_diff, n_act, err, mab))
    assert n_diff <= 1e-3 * max(n_act, 1)
    assert err <= 1e-2 and mab <= 2e-2


@pytest.mark.parametrize("cfg", CASES, ids=_cid)
def test_layer_nvfp4_vs_oracle(cfg):
    toks = np.arange(cfg.T) if cfg.T <= 64 else np.unique(np.linspace(0, cfg.T - 1, 24).astype(np.int64))
    check_layer_nvfp4(cfg, toks)


def test_layer_nvfp4_dense_gemm2_path():
    check_layer_nvfp4(SMALL, np.arange(0, SMALL.T, 9), path=moe.GEMM2_DENSE)


def test_layer_nvfp4_full_prefill():
    cfg = synth.CONFIGS["prefill_t32768"]
    rng = np.random.default_rng(7)
    toks = np.unique(np.concatenate([[0, cfg.T - 1], rng.choice(cfg.T, 30, replace=False)]))
    check_layer_nvfp4(cfg, toks)


def test_layer_nvfp4_refuses_decode_tilings():
    cfg = SMALL.replace(block_n=32)
    shape = shape_of(cfg)
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    g = torch.ones(cfg.E_local, dtype=torch.float32, device="cuda")
    nv = moe.MoeNvfp4(X_GS, H_GS, g, g)
    x, logits, sl = device_inputs(cfg)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_nvfp4(shape, nv, logits, sl, x, moe.MoeWeights(dummy, dummy, dummy, dummy), moe.workspace(shape))
    assert e.value.rc == moe.MOE_ERR_SHAPE
