"""The GEMM2 gate and its two paths, through the C ABI (marked gpu).

"[FlashInfer] Device-side gating for the MoE GEMM2 path": a device-side
decision, taken once the sorted row count is known (here by the sort's
placement thread, in the launch that writes the table's header), picks split
(FC2 writes each routed row, the combine sums a token's rows) or dense (FC2's
epilogue reduces w * Y into an fp32 [T, H] accumulator, the combine converts
it), in one fixed launch chain.  Each path
is forced through the gate here and must meet the layer's output bar against
the oracle (relative L2 <= 1e-2, max-abs <= 2e-2; the page itself accepts a
different summation order between the paths).  The gate's own rule is
checked on the workloads, and the path a call took is read back from the
workspace header."""
import numpy as np
import pytest
import torch

import mxfp4_mixture_experts_02_gb300 as moe
import synth
from moe_case import (OracleCase, bf16_bits, bf16_to_f64, dense_repeat_bound, device_inputs, device_weights, rel_l2,
                       shape_of, within_dense_repeat)

pytestmark = pytest.mark.gpu

SMALL = synth.MoeConfig("small", 7, T=48, E_global=64, E_local=64, expert_offset=0, top_k=4, num_shared=0,
                        hidden=1024, inter=256, block_n=32)

CASES = [
    SMALL.replace(T=7, block_n=16),
    SMALL.replace(T=96, block_n=32, num_shared=1, zipf_s=1.1),
    SMALL.replace(T=600, block_n=32, num_shared=1, zipf_s=1.1),  # route, sort and x as separate launches
    SMALL.replace(T=200, block_n=128, top_k=8, num_shared=1),
    SMALL.replace(T=256, block_n=16, E_local=32, expert_offset=16),  # EP slice: tokens without local rows
    synth.CONFIGS["tiny"],
    # every token on experts 0 .. k-1 (Zipf s = 30): the dense path's
    # reductions of four experts' tiles all land on the same token rows
    SMALL.replace(T=600, block_n=32, zipf_s=30.0),
    SMALL.replace(T=1000, block_n=128, num_shared=1, zipf_s=30.0),
]


def _cid(c):
    return "%s-T%d-B%d-E%d+%d-S%d" % (c.name, c.T, c.block_n, c.E_local, c.expert_offset, c.num_shared)


def run_path(cfg, path, tokens):
    shape = shape_of(cfg)
    wts = device_weights(cfg)
    x, logits, sl = device_inputs(cfg)
    ws = moe.workspace(shape)
    moe.moe_set_gemm2_path(path)
    try:
        out, _, _ = moe.moe_layer(shape, logits, sl, x, wts, ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_gemm2_path(moe.GEMM2_AUTO)
    assert moe.moe_get_status(ws) == (0, 0)
    took = int(moe.moe_get_views(shape, ws)["header"][5].item())
    return bf16_to_f64(bf16_bits(out)[tokens]), took


@pytest.mark.parametrize("cfg", CASES + [synth.CONFIGS[n] for n in ("decode_t32", "ep_slice_t64",
                                                                     "skewed_shared_t256", "prefill_t32768")],
                         ids=_cid)
def test_both_gemm2_paths_match_the_oracle(cfg):
    toks = np.arange(cfg.T) if cfg.T <= 64 else np.unique(np.linspace(0, cfg.T - 1, 24).astype(np.int64))
    ref = OracleCase(cfg).forward(toks)["out_f64"]
    res = {}
    for path, code in ((moe.GEMM2_SPLIT, 0), (moe.GEMM2_DENSE, 1)):
        got, took = run_path(cfg, path, toks)
        assert took == code
        err, mab = rel_l2(got, ref), float(np.max(np.abs(got - ref)))
        res[code] = (err, mab)
        assert err <= 1e-2 and mab <= 2e-2, (path, err, mab)
    print("GATE %s split rel_l2=%.3g max_abs=%.3g dense rel_l2=%.3g max_abs=%.3g" % (
        _cid(cfg), res[0][0], res[0][1], res[1][0], res[1][1]))


def test_gate_rule_on_the_workloads():
    # dense where the [T, H] fp32 accumulator is at most 32 MiB (every decode
    # workload), split at the 32768-token prefill
    want = {"tiny": 1, "decode_t32": 1, "ep_slice_t64": 1, "skewed_shared_t256": 1, "prefill_t32768": 0}
    for name, path in want.items():
        cfg = synth.CONFIGS[name]
        shape = shape_of(cfg)
        ws = moe.workspace(shape)
        x, logits, sl = device_inputs(cfg)
        moe.moe_layer(shape, logits, sl, x, device_weights(cfg), ws)
        torch.cuda.synchronize()
        assert int(moe.moe_get_views(shape, ws)["header"][5].item()) == path, name


@pytest.mark.parametrize("T,block_n,path", [(2340, 32, 1), (2341, 32, 0), (2340, 16, 1), (1024, 128, 1),
                                            (1025, 128, 0)])
def test_gate_rule_boundaries(T, block_n, path):
    # at the layer's shape (H 3584, 896 experts, top-16): the fp32 accumulator
    # is 32 MiB at T 2340, one token more leaves L2 (split at every tiling);
    # the 128-row tiling's rows * H reaches 56 Mi at T 1024 (R = 16 T)
    shape = moe.MoeShape(T=T, max_T=T, E_global=896, E_local=896, expert_offset=0, top_k=16, num_shared=0,
                         hidden=3584, inter=384, block_n=block_n)
    rng = np.random.default_rng(T)
    ids = np.argsort(rng.random((T, 896)), axis=1)[:, :16].astype(np.int32)  # 16 distinct experts per token
    ws = moe.workspace(shape)
    moe.moe_sort(shape, torch.from_numpy(ids).cuda(), ws)
    torch.cuda.synchronize()
    hdr = moe.moe_get_views(shape, ws)["header"].cpu().numpy()
    assert hdr[0] == 16 * T and hdr[5] == path


@pytest.mark.parametrize("cfg", [CASES[0], CASES[2], CASES[3]], ids=_cid)
def test_dense_path_repeats_within_its_bound(cfg):
    # the dense path's reductions run in no fixed order: two calls agree to
    # within one bf16 step of the output plus the fp32 reordering error of the
    # token's terms, bounded from the split path's rows (dense_repeat_bound;
    # the split path is bit-reproducible, tested with graph replay)
    shape = shape_of(cfg)
    wts = device_weights(cfg)
    x, logits, sl = device_inputs(cfg)
    ws = moe.workspace(shape)
    outs = []
    for path in (moe.GEMM2_SPLIT, moe.GEMM2_DENSE, moe.GEMM2_DENSE):
        moe.moe_set_gemm2_path(path)
        try:
            out, _, _ = moe.moe_layer(shape, logits, sl, x, wts, ws)
            torch.cuda.synchronize()
        finally:
            moe.moe_set_gemm2_path(moe.GEMM2_AUTO)
        assert moe.moe_get_status(ws) == (0, 0)
        if path == moe.GEMM2_SPLIT:
            slack = dense_repeat_bound(shape, ws, cfg.T)
        else:
            outs.append(out.double().cpu().numpy())
    assert within_dense_repeat(outs[0], outs[1], slack)
