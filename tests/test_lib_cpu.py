"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every function include/moe_api.h declares, and rejects bad arguments on the
host (no kernel launch) with the documented error codes."""
import ctypes
import os
import re

import pytest

import mxfp4_mixture_experts_02_gb300 as moe
from conftest import ROOT


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_api.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*int\s+(moe_\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_symbol():
    L = moe.lib()
    names = _declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n


def _shape(**kw):
    base = dict(T=32, max_T=32, E_global=896, E_local=896, expert_offset=0, top_k=16, num_shared=0, hidden=3584,
                inter=384, block_n=32)
    base.update(kw)
    return moe.MoeShape(**base)


def test_supported_shapes_and_limits():
    assert moe.moe_is_supported(_shape())
    assert moe.moe_is_supported(_shape(block_n=16, E_local=448, expert_offset=448, T=64, max_T=64))
    assert moe.moe_is_supported(_shape(num_shared=1, T=256, max_T=256))
    assert moe.moe_is_supported(_shape(activation=moe.ACT_SWIGLU_CLAMP, act_params=(7.0, 0.0)))
    assert moe.moe_is_supported(_shape(activation=moe.ACT_SITU, act_params=(4.0, 25.0)))
    bad = [dict(hidden=3500), dict(hidden=256), dict(inter=192), dict(block_n=64), dict(block_n=8),
           dict(top_k=0), dict(top_k=33), dict(top_k=900, E_global=896), dict(E_global=2048, E_local=2048),
           dict(num_shared=2), dict(E_local=0), dict(expert_offset=448), dict(expert_offset=-1),
           dict(T=33), dict(T=-1), dict(max_T=1 << 20), dict(activation=3), dict(activation=-1),
           dict(activation=1), dict(activation=1, act_params=(-1.0, 0.0)),
           dict(activation=1, act_params=(float("inf"), 0.0)), dict(activation=1, act_params=(float("nan"), 0.0)),
           dict(activation=2, act_params=(4.0, 0.0)), dict(activation=2, act_params=(0.0, 25.0))]
    for kw in bad:
        assert not moe.moe_is_supported(_shape(**kw)), kw


def test_workspace_bytes_grows_with_max_tokens():
    a = moe.moe_workspace_bytes(_shape(T=1, max_T=32))
    b = moe.moe_workspace_bytes(_shape(T=1, max_T=256))
    assert 0 < a < b
    with pytest.raises(moe.MoeError) as e:
        moe.moe_workspace_bytes(_shape(hidden=100))
    assert e.value.rc == -2


def test_host_side_errors_launch_nothing():
    L = moe.lib()
    s = _shape().c()
    # NULL pointers
    assert L.moe_route(ctypes.byref(s), None, None, None, None, None) == -1
    assert L.moe_sort(ctypes.byref(s), None, None, 0, None) == -1
    assert L.moe_get_status(None, None, None) == -1
    # unsupported shape
    bad = _shape(block_n=64).c()
    assert L.moe_sort(ctypes.byref(bad), 16, 256, 1 << 30, None) == -2
    # workspace misaligned / too small (checked before any launch)
    assert L.moe_sort(ctypes.byref(s), 16, 255, 1 << 30, None) == -3
    assert L.moe_sort(ctypes.byref(s), 16, 256, 100, None) == -4
    # misaligned weights
    w = moe.lib  # noqa: F841
    from mxfp4_mixture_experts_02_gb300 import _Weights
    wt = _Weights(48, 256, 256, 256)  # w1 not 32-byte aligned
    need = moe.moe_workspace_bytes(_shape())
    assert L.moe_forward(ctypes.byref(s), 256, ctypes.byref(wt), 256, 256, need, 256, None) == -3
    # router entry points: NULL, unsupported shape, misaligned buffers, small workspace
    need = moe.moe_workspace_bytes(_shape())
    assert L.moe_router(ctypes.byref(s), None, 256, 256, 256, need, None) == -1
    assert L.moe_router(ctypes.byref(bad), 256, 256, 256, 256, need, None) == -2
    assert L.moe_router(ctypes.byref(s), 264, 256, 256, 256, need, None) == -3  # x not 16-byte aligned
    assert L.moe_router(ctypes.byref(s), 256, 256, 260, 256, need, None) == -3  # logits not 16-byte aligned
    assert L.moe_router(ctypes.byref(s), 256, 256, 256, 256, 100, None) == -4
    assert L.moe_layer_router(ctypes.byref(s), None, None, 256, ctypes.byref(wt), 256, 256, 256, 256, need, 256,
                              None) == -1
    good = _Weights(256, 256, 256, 256)
    assert L.moe_layer_router(ctypes.byref(s), 256, None, 256, ctypes.byref(good), 256, 256, 256, 256, 100, 256,
                              None) == -4
    # packing size rules
    assert L.moe_pack_weights(16, 16, 2, 100, 128, 0, 16, 16, None) == -2
    assert L.moe_pack_weights(16, 16, 2, 128, 128, 1, 16, 16, None) == -2
    assert L.moe_quantize_mxfp4(16, 4, 33, 16, 16, None) == -2


def test_packed_weight_sizes():
    # 256-row blocks; packed sizes equal the row-major inputs'
    assert moe.moe_packed_weight_bytes(2, 3584, 384, False) == (256, 2 * 3584 * 192, 2 * 3584 * 12)
    assert moe.moe_packed_weight_bytes(3, 768, 3584, True) == (256, 3 * 768 * 1792, 3 * 768 * 112)
    for bad in [(2, 100, 384, False), (2, 448, 384, True), (2, 512, 100, False), (0, 512, 384, False)]:
        with pytest.raises(moe.MoeError):
            moe.moe_packed_weight_bytes(*bad)


def test_gemm2_path_override_checks_its_value():
    for path in (moe.GEMM2_SPLIT, moe.GEMM2_DENSE, moe.GEMM2_AUTO):
        moe.moe_set_gemm2_path(path)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_set_gemm2_path(3)
    assert e.value.rc == moe.MOE_ERR_SHAPE


def test_layer_launch_count():
    # decode: route + sort + x quantisation in one launch (the GEMM2 gate decided
    # in it), FC1, FC2, combine
    assert moe.moe_layer_launch_count(_shape()) == 4
    # up to 64 tokens the decode tilings route, sort and quantise x in one cluster launch;
    # up to 512 x rides on the route launch and a one-CTA sort follows
    assert moe.moe_layer_launch_count(_shape(T=64, max_T=64)) == 4
    assert moe.moe_layer_launch_count(_shape(T=65, max_T=65)) == 5
    assert moe.moe_layer_launch_count(_shape(T=512, max_T=512)) == 5
    # 513 tokens: route, one-CTA sort, x quantisation, FC1, FC2, combine
    assert moe.moe_layer_launch_count(_shape(T=513, max_T=513)) == 6
    # prefill tiling at 32768 tokens: route, 3-kernel sort, gather, FC1, FC2, combine
    assert moe.moe_layer_launch_count(_shape(T=32768, max_T=32768, block_n=128)) == 8
    assert moe.moe_layer_launch_count(_shape(T=0)) == 1

