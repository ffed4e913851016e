"""The device-error path through the C ABI (marked gpu).

Every wait in the GEMM kernels is bounded; on expiry the CTA records
MOE_ERR_TIMEOUT and the site in the workspace status word, stops its other
roles, lets the copies it issued land, frees its tensor memory and exits, so
the context stays usable.  moe_test_set_stall makes one such wait run out on
demand: the FC1 MMA thread waits on a barrier that nothing arrives on.  The
call must report the timeout, and the next call on the same workspace must be
clean and give the normal result."""
import pytest
import torch

import mxfp4_mixture_experts_02_gb300 as moe
import synth
from moe_case import device_inputs, device_weights, shape_of

pytestmark = pytest.mark.gpu

SMALL = synth.MoeConfig("small", 7, T=48, E_global=64, E_local=64, expert_offset=0, top_k=4, num_shared=0,
                        hidden=1024, inter=256, block_n=32)


@pytest.fixture
def split_path():
    # the clean call is compared bit for bit: the split GEMM2 path sums in a
    # fixed order (the dense path does not)
    moe.moe_set_gemm2_path(moe.GEMM2_SPLIT)
    yield
    moe.moe_set_gemm2_path(moe.GEMM2_AUTO)


@pytest.mark.parametrize("cfg", [SMALL, SMALL.replace(T=200, block_n=128, num_shared=1)], ids=["decode", "prefill"])
def test_expired_wait_is_reported_and_the_next_call_is_clean(cfg, split_path):
    shape = shape_of(cfg)
    wts = device_weights(cfg)
    x, logits, sl = device_inputs(cfg)
    ref, _, _ = moe.moe_layer(shape, logits, sl, x, wts, moe.workspace(shape))
    ws = moe.workspace(shape)
    moe.moe_test_set_stall(2_000_000)  # 2 ms
    try:
        moe.moe_layer(shape, logits, sl, x, wts, ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_test_set_stall(0)
    st, detail = moe.moe_get_status(ws)
    assert st == moe.MOE_ERR_TIMEOUT, (st, detail)
    assert detail >> 16 == 5, detail  # the stall site
    assert 0 <= (detail & 0xFFFF) < moe.moe_num_sms()  # the block that recorded it
    out, _, _ = moe.moe_layer(shape, logits, sl, x, wts, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_status(ws) == (0, 0)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
