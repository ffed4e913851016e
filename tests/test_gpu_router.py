"""Router GEMM (x bf16 times the bf16 router matrix -> fp32 logits) and the
layer chain that starts from it, against the oracle, through the C ABI.

Bars:
  - logits: |gpu - oracle| <= (H / 8) * 2^-23 * sum_h |x_h w_h| per element
    (fp32 accumulation of exact bf16 products in another order; the bound is
    H/8 roundings of the absolute sum) and relative L2 <= 1e-5; repeated runs
    bit-identical (fixed-order split-K sums);
  - ids: equal to the oracle's top-k of its own logits, except at near ties
    (the k-th and (k+1)-th oracle logits closer than the logits bound), where
    the GPU's pick must still be a valid top-k within that bound;
  - output on sampled tokens (with identical ids): relative L2 <= 1e-2 and
    max-abs <= 2e-2 against the fp64 oracle.
"""
import math

import numpy as np
import pytest
import torch

import mxfp4_mixture_experts_02_gb300 as moe
import oracle
import synth
from moe_case import OracleCase, bf16_bits, bf16_to_f64, device_weights, rel_l2, router_matrix_bits, shape_of

pytestmark = pytest.mark.gpu

BASE = synth.MoeConfig("router", 21, T=32, E_global=896, E_local=896, expert_offset=0, top_k=16, num_shared=0,
                       hidden=3584, inter=384, block_n=32, router="matrix")


def _cfg(T, Eg, H, **kw):
    c = BASE.replace(T=T, E_global=Eg, E_local=Eg, hidden=H, router_sigma=1.0 / math.sqrt(H), **kw)
    return c.replace(top_k=min(c.top_k, Eg))


def _bound(x_bits, wr_bits):
    x = bf16_to_f64(x_bits)
    w = bf16_to_f64(wr_bits)
    H = x.shape[1]
    return (H / 8.0) * 2.0 ** -23 * (np.abs(x) @ np.abs(w).T)


def _run_router(cfg):
    shape = shape_of(cfg)
    x = synth.x_device(cfg)
    wr_bits = router_matrix_bits(cfg)
    wr = torch.from_numpy(wr_bits.view(np.int16)).cuda().view(torch.bfloat16)
    ws = moe.workspace(shape)
    lg = moe.moe_router(shape, x, wr, ws)
    lg2 = moe.moe_router(shape, x, wr, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_status(ws) == (0, 0)
    return lg.cpu().numpy(), lg2.cpu().numpy(), wr_bits


@pytest.mark.parametrize("T,Eg,H", [(32, 896, 3584), (1, 64, 512), (7, 33, 1024), (200, 896, 1024),
                                    (300, 896, 3584), (1200, 100, 1536)])
def test_router_logits_vs_oracle(T, Eg, H):
    cfg = _cfg(T, Eg, H)
    got, again, wr_bits = _run_router(cfg)
    np.testing.assert_array_equal(got, again)
    rows = np.arange(T) if T <= 64 else np.unique(np.concatenate([[0, T - 1], np.random.default_rng(T).choice(T, 30)]))
    x_bits = synth.x_host(cfg)[rows]
    ref = oracle.router_logits(x_bits, wr_bits)
    err = np.abs(got[rows].astype(np.float64) - ref)
    bound = _bound(x_bits, wr_bits)
    assert np.all(err <= bound), float(np.max(err / bound))
    assert rel_l2(got[rows], ref) <= 1e-5


def _near_tie_ok(got_ids, ref_logits, k, tol):
    """The GPU's k picks are a valid top-k of the oracle logits within tol."""
    order = np.sort(ref_logits)[::-1]
    kth = order[k - 1]
    return all(ref_logits[e] >= kth - 2 * tol for e in got_ids[:k])


@pytest.mark.parametrize("T,block_n", [(32, 32), (300, 128)])
def test_layer_from_router_matrix_vs_oracle(T, block_n):
    cfg = _cfg(T, 896, 3584, block_n=block_n)
    shape = shape_of(cfg)
    wts = device_weights(cfg)
    x = synth.x_device(cfg)
    wr_bits = router_matrix_bits(cfg)
    wr = torch.from_numpy(wr_bits.view(np.int16)).cuda().view(torch.bfloat16)
    ws = moe.workspace(shape)
    out, lg, ids, w = moe.moe_layer_router(shape, wr, None, x, wts, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_status(ws) == (0, 0)
    x_bits = synth.x_host(cfg)
    ref_lg = oracle.router_logits(x_bits, wr_bits)
    bound = _bound(x_bits, wr_bits)
    got_lg = lg.cpu().numpy()
    assert np.all(np.abs(got_lg.astype(np.float64) - ref_lg) <= bound)
    orc = OracleCase(cfg, logits=ref_lg)
    gids = ids.cpu().numpy()
    same = np.all(gids == orc.ids, axis=1)
    for t in np.nonzero(~same)[0]:
        assert _near_tie_ok(gids[t], ref_lg[t].astype(np.float64), cfg.top_k, float(np.max(bound[t]))), t
    assert same.mean() >= 0.99
    toks = np.nonzero(same)[0]
    toks = toks if toks.size <= 6 else np.unique(np.concatenate([toks[:2], toks[-2:], toks[toks.size // 2:][:2]]))
    ref = orc.forward(toks)
    got = bf16_to_f64(bf16_bits(out)[toks])
    assert rel_l2(got, ref["out_f64"]) <= 1e-2
    assert np.max(np.abs(got - ref["out_f64"])) <= 2e-2
