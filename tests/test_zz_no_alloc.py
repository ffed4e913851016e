"""moe_layer_noalloc: the layer for callers that cannot allocate device memory
(code running under an allocator that forbids new allocations, runtimes that
must not call cudaMalloc after start-up).  Its scratch is the library's fixed
32 MiB device array, shared by every call on a device and left holding the
previous call's contents.  These tests run it on three shapes in a row (a
larger one, a smaller one, the larger one again, so stale maps and rows of an
earlier call are present) and require, after each call, exactly the result
of moe_layer on a fresh caller workspace -- both run the same kernels on the
same inputs -- and a clean status word; shapes needing more scratch are
refused.

This file is collected last so that a run stopping at its first failure has
already run every other test."""
import pytest
import torch

import mxfp4_mixture_experts_02_gb300 as moe
import synth
from moe_case import device_inputs, device_weights, shape_of

pytestmark = pytest.mark.gpu

SMALL = synth.MoeConfig("small", 7, T=48, E_global=64, E_local=64, expert_offset=0, top_k=4, num_shared=1,
                        hidden=1024, inter=256, block_n=16, shared_scale=0.5)


@pytest.fixture
def split_path():
    # exact equality needs the bit-reproducible GEMM2 path (the dense one sums
    # in no fixed order)
    moe.moe_set_gemm2_path(moe.GEMM2_SPLIT)
    yield
    moe.moe_set_gemm2_path(moe.GEMM2_AUTO)


def test_noalloc_matches_workspace_entry_point_across_calls(split_path):
    cases = {}
    for cfg in (SMALL, synth.CONFIGS["tiny"]):
        shape = shape_of(cfg)
        wts = device_weights(cfg)
        x, logits, sl = device_inputs(cfg)
        ws = moe.workspace(shape)
        ref = moe.moe_layer(shape, logits, sl, x, wts, ws)
        torch.cuda.synchronize()
        assert moe.moe_get_status(ws) == (0, 0)
        cases[cfg.name] = (shape, wts, x, logits, sl, ref)
    for name in ("small", "tiny", "small"):
        shape, wts, x, logits, sl, (ref_out, ref_ids, ref_w) = cases[name]
        out, ids, w = moe.moe_layer_noalloc(shape, logits, sl, x, wts)
        torch.cuda.synchronize()
        assert moe.moe_noalloc_get_status() == (0, 0), name
        assert torch.equal(ids, ref_ids), name
        assert torch.equal(w, ref_w), name
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), name


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
