"""moe_layer_noalloc: the layer for callers that cannot allocate device memory
(code running under an allocator that forbids new allocations, runtimes that
must not call cudaMalloc after start-up).  Its scratch is the library's fixed
32 MiB device array, so these tests compare it with moe_layer on a caller
workspace, call it twice in a row (the array keeps the previous call's
contents), and check that shapes needing more scratch are refused.

This file is collected last so that a run stopping at its first failure has
already run every other test."""
import numpy as np
import pytest
import torch

import mxfp4_mixture_experts_02_gb300 as moe
import synth
from moe_case import bf16_bits, bf16_to_f64, device_inputs, device_weights, rel_l2, shape_of

pytestmark = pytest.mark.gpu

SMALL = synth.MoeConfig("small", 7, T=48, E_global=64, E_local=64, expert_offset=0, top_k=4, num_shared=1,
                        hidden=1024, inter=256, block_n=16, shared_scale=0.5)


@pytest.mark.parametrize("cfg", [SMALL, synth.CONFIGS["tiny"]], ids=["small", "tiny"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(cfg):
    shape = shape_of(cfg)
    wts = device_weights(cfg)
    x, logits, sl = device_inputs(cfg)
    ws = moe.workspace(shape)
    ref, ref_ids, ref_w = moe.moe_layer(shape, logits, sl, x, wts, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_status(ws) == (0, 0)
    ref_f = bf16_to_f64(bf16_bits(ref))
    for _ in range(2):
        out, ids, w = moe.moe_layer_noalloc(shape, logits, sl, x, wts)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids)
        np.testing.assert_allclose(w.cpu().numpy(), ref_w.cpu().numpy(), rtol=4e-6, atol=1e-7)
        got = bf16_to_f64(bf16_bits(out))
        assert rel_l2(got, ref_f) <= 1e-2
        assert np.max(np.abs(got - ref_f)) <= 2e-2


def test_noalloc_refuses_shapes_beyond_its_scratch():
    cfg = synth.CONFIGS["skewed_shared_t256"]  # needs ~96 MiB of workspace
    shape = shape_of(cfg)
    assert moe.moe_workspace_bytes(shape) > 32 << 20
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    wts = moe.MoeWeights(dummy, dummy, dummy, dummy)
    x = torch.zeros((cfg.T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros((cfg.T, cfg.E_global), dtype=torch.float32, device="cuda")
    sl = torch.zeros((cfg.T, 1), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_noalloc(shape, lg, sl, x, wts)
    assert e.value.rc == moe.MOE_ERR_WORKSPACE
