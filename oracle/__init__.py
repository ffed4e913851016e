"""CPU oracle for the fused MXFP4 MoE layer forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It wraps ``moe_oracle.cpp`` (plain C++17, fp64,
brute force), which shares no code with the GPU library.

Functions and the passages they follow (reference page titles):
  router_logits -- fp32(sum_h x[t,h] * wr[e,h]) of bf16 x and router rows
                (the router GEMM in front of the routing step).
  route      -- top-k with renormalised softmax weights; the shared expert's
                weight sigmoid(fp32(logit)) * scale ("[sglang] SGLang MoE
                shared expert: fuse 3 kernels into 1", kernel change).
  sort       -- prepare_moe_input's expert_offsets / a_map / c_map ("[SGLang]
                CUTLASS MoE", section 1) and the virtual experts of kBlockN rows
                ("[sglang] ... MXFP4 decode MoE ... shape templates",
                sections 1 and 5, including the expert_offset slice).
  forward    -- the dataflow of the "[SGLang] CUTLASS MoE" structure diagram
                with MXFP8 activations, MXFP4 weights, silu_and_mul (section 4)
                and apply_shuffle_mul_sum (section 5); the FC1 activation may
                instead be the clamped SwiGLU or SiTU of "... MXFP4 decode MoE
                ... shape templates", section 4.
  activation -- h(gate, up) of one element, fp64.
  quantize_* -- the OCP MX v1.0 conversion rule for E2M1 / E4M3 blocks of 32.
  nvfp4_*, quantize_nvfp4*, forward_nvfp4
             -- the FP4 variant of "[SGLang] CUTLASS MoE", section 6: E2M1
                with one E4M3 scale per 16 elements and an fp32 global scale
                per tensor (value = e2m1 * e4m3 / gs), and the layer forward
                with NVFP4 activations and weights.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

FMT_E2M1 = 0
FMT_E4M3 = 1
ACT_SWIGLU = 0
ACT_SWIGLU_CLAMP = 1
ACT_SITU = 2


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + ".tmp%d" % os.getpid()
    cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-o", tmp, _SRC]
    subprocess.check_call(cmd)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.oracle_e2m1_value.restype = dbl
        L.oracle_e2m1_value.argtypes = [i32]
        L.oracle_e4m3_value.restype = dbl
        L.oracle_e4m3_value.argtypes = [i32]
        L.oracle_e8m0_value.restype = dbl
        L.oracle_e8m0_value.argtypes = [i32]
        L.oracle_bf16_rne.restype = ctypes.c_uint16
        L.oracle_bf16_rne.argtypes = [dbl]
        L.oracle_activation.restype = dbl
        L.oracle_activation.argtypes = [i32, dbl, dbl, dbl, dbl]
        L.oracle_mx_quantize_block.restype = None
        L.oracle_mx_quantize_block.argtypes = [P, i32, i32, P, P]
        L.oracle_quantize_mxfp4.restype = None
        L.oracle_quantize_mxfp4.argtypes = [P, i64, i64, P, P]
        L.oracle_quantize_mxfp8_bf16.restype = None
        L.oracle_quantize_mxfp8_bf16.argtypes = [P, i64, i64, P, P]
        L.oracle_router_logits.restype = None
        L.oracle_router_logits.argtypes = [i32, i32, i32, P, P, P]
        L.oracle_route.restype = None
        L.oracle_route.argtypes = [i32, i32, i32, P, i32, P, dbl, P, P]
        L.oracle_sort.restype = i32
        L.oracle_sort.argtypes = [i32, i32, P, i32, i32, i32, i32, i32, P, P, P, P, P]
        L.oracle_forward.restype = i32
        L.oracle_forward.argtypes = [i32] * 8 + [P] * 8 + [i32] + [P] * 7 + [i32, dbl, dbl, P]
        flt = ctypes.c_float
        L.oracle_nvfp4_quantize_block.restype = None
        L.oracle_nvfp4_quantize_block.argtypes = [P, flt, P, P]
        L.oracle_nvfp4_global_scale.restype = flt
        L.oracle_nvfp4_global_scale.argtypes = [P, i64]
        L.oracle_quantize_nvfp4.restype = None
        L.oracle_quantize_nvfp4.argtypes = [P, i64, i64, flt, P, P]
        L.oracle_quantize_nvfp4_bf16.restype = None
        L.oracle_quantize_nvfp4_bf16.argtypes = [P, i64, i64, flt, P, P]
        L.oracle_forward_nvfp4.restype = i32
        L.oracle_forward_nvfp4.argtypes = ([i32] * 8 + [P] * 4 + [P] * 6 + [flt, flt, i32] + [P] * 7 +
                                           [i32, dbl, dbl, P])
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ formats
def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(int(code))


def e8m0_value(code: int) -> float:
    return lib().oracle_e8m0_value(int(code))


def bf16_rne(d: float) -> int:
    return int(lib().oracle_bf16_rne(float(d)))


def activation(act: int, params, g: float, u: float) -> float:
    """h(g, u) of the FC1 epilogue; params = (limit,) or (beta, linear_beta)."""
    c = (list(params) + [0.0, 0.0])[:2]
    return lib().oracle_activation(int(act), float(c[0]), float(c[1]), float(g), float(u))


def mx_quantize_block(values, fmt: int):
    """One MX block (any length): returns (codes uint8[n], scale_code int)."""
    v = _c(values, np.float64)
    codes = np.zeros(v.size, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib().oracle_mx_quantize_block(_p(v), v.size, fmt, _p(codes), _p(sc))
    return codes, int(sc[0])


def quantize_mxfp4(w):
    """fp32 [rows, K] -> (packed E2M1 codes uint8 [rows, K/2], E8M0 uint8 [rows, K/32])."""
    w = _c(w, np.float32)
    rows, K = w.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    scales = np.zeros((rows, K // 32), np.uint8)
    lib().oracle_quantize_mxfp4(_p(w), rows, K, _p(codes), _p(scales))
    return codes, scales


def quantize_mxfp8_bf16(x_bits):
    """bf16 bits uint16 [rows, K] -> (E4M3 codes uint8 [rows, K], E8M0 uint8 [rows, K/32])."""
    x = _c(x_bits, np.uint16)
    rows, K = x.shape
    codes = np.zeros((rows, K), np.uint8)
    scales = np.zeros((rows, K // 32), np.uint8)
    lib().oracle_quantize_mxfp8_bf16(_p(x), rows, K, _p(codes), _p(scales))
    return codes, scales


# ------------------------------------------------------------------ routing
def router_logits(x_bits, wr_bits):
    """bf16 bits x [T, H], router rows wr [Eg, H] -> fp32 logits [T, Eg]."""
    x = _c(x_bits, np.uint16)
    wr = _c(wr_bits, np.uint16)
    T, H = x.shape
    Eg = wr.shape[0]
    assert wr.shape[1] == H
    out = np.zeros((T, Eg), np.float32)
    lib().oracle_router_logits(T, H, Eg, _p(x), _p(wr), _p(out))
    return out


def route(logits, top_k: int, num_shared: int = 0, shared_logit=None, shared_scale: float = 1.0):
    """logits fp32 [T, Eg] -> (ids int32 [T, k+S], weights float64 [T, k+S])."""
    lg = _c(logits, np.float32)
    T, Eg = lg.shape
    kp = top_k + num_shared
    ids = np.zeros((T, kp), np.int32)
    w = np.zeros((T, kp), np.float64)
    sl = None if num_shared == 0 else _c(shared_logit, np.uint16).reshape(T, num_shared)
    lib().oracle_route(T, Eg, top_k, _p(lg), num_shared, _p(sl), float(shared_scale), _p(ids), _p(w))
    return ids, w


def sort(ids, E_global: int, E_local: int, expert_offset: int, num_shared: int, block_n: int):
    """ids int32 [T, k'] -> dict with counts, offsets, a_map, c_map, vinfo [num_v, 4], num_v."""
    ids = _c(ids, np.int32)
    T, kp = ids.shape
    Et = E_local + num_shared
    counts = np.zeros(Et, np.int32)
    offsets = np.zeros(Et + 1, np.int32)
    c_map = np.zeros(T * kp, np.int32)
    a_map = np.full(T * kp, -1, np.int32)
    vmax = Et + (T * kp) // block_n + 1
    vinfo = np.zeros((vmax, 4), np.int32)
    nv = lib().oracle_sort(T, kp, _p(ids), E_global, E_local, expert_offset, num_shared, block_n,
                           _p(counts), _p(offsets), _p(a_map), _p(c_map), _p(vinfo))
    R = int(offsets[-1])
    return dict(counts=counts, offsets=offsets, a_map=a_map[:R].copy(), c_map=c_map,
                vinfo=vinfo[:nv].copy(), num_v=int(nv))


# ------------------------------------------------------------------ forward
def forward(x_bits, ids, w, wmap, w1, w1s, w2, w2s, *, H: int, I: int, E_global: int, E_local: int,
            expert_offset: int, num_shared: int, tokens=None, want_act: bool = False, want_xq: bool = False,
            activation: int = ACT_SWIGLU, act_params=(0.0, 0.0), want_y: bool = False):
    """Layer forward for ``tokens`` (default: all).

    x_bits uint16 [T, H] (bf16); ids int32 [T, k']; w float64 [T, k'];
    wmap int32 [E_local + S] -> index into the compact weight arrays
    w1 [n, 2I, H/2], w1s [n, 2I, H/32], w2 [n, H, I/2], w2s [n, H, I/32].
    activation / act_params select the FC1 activation (see ``activation``).
    Returns dict(out_f64, out_bf16 (uint16 bits), [act, act_sf], [xq, xq_sf],
    [y_slot float64 [n, k', H]: each slot's w * Y, the rows the un-permute sums]).
    """
    x = _c(x_bits, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    T, kp = ids.shape
    toks = _c(np.arange(T) if tokens is None else tokens, np.int32)
    n = toks.size
    out = np.zeros((n, H), np.float64)
    outb = np.zeros((n, H), np.uint16)
    act = np.zeros((n, kp, I), np.uint8) if want_act else None
    acts = np.zeros((n, kp, I // 32), np.uint8) if want_act else None
    xq = np.zeros((n, H), np.uint8) if want_xq else None
    xqs = np.zeros((n, H // 32), np.uint8) if want_xq else None
    ys = np.zeros((n, kp, H), np.float64) if want_y else None
    arrs = [_c(a, np.uint8) for a in (w1, w1s, w2, w2s)]
    wm = _c(wmap, np.int32)
    c = (list(act_params) + [0.0, 0.0])[:2]
    rc = lib().oracle_forward(T, H, I, kp, E_global, E_local, expert_offset, num_shared, _p(x), _p(ids), _p(w),
                              _p(wm), *[_p(a) for a in arrs], n, _p(toks), _p(out), _p(outb), _p(act), _p(acts),
                              _p(xq), _p(xqs), int(activation), float(c[0]), float(c[1]), _p(ys))
    if rc != 0:
        raise ValueError("oracle_forward: a routed expert has no weights in wmap")
    res = dict(out_f64=out, out_bf16=outb)
    if want_act:
        res.update(act=act, act_sf=acts)
    if want_xq:
        res.update(xq=xq, xq_sf=xqs)
    if want_y:
        res.update(y_slot=ys)
    return res


# ------------------------------------------------------------------ NVFP4
def nvfp4_quantize_block(values, gs: float):
    """One NVFP4 block of 16 fp32 values with global scale gs: (E2M1 codes
    uint8[16] with the sign in bit 3, E4M3 scale code)."""
    v = _c(values, np.float32)
    assert v.size == 16
    codes = np.zeros(16, np.uint8)
    sf = np.zeros(1, np.uint8)
    lib().oracle_nvfp4_quantize_block(_p(v), float(gs), _p(codes), _p(sf))
    return codes, int(sf[0])


def nvfp4_global_scale(w) -> float:
    """fp32(2688 / amax) of a weight matrix (1 for all zeros)."""
    w = _c(w, np.float32)
    return float(lib().oracle_nvfp4_global_scale(_p(w), w.size))


def quantize_nvfp4(w, gs: float):
    """fp32 [rows, K] -> (packed E2M1 codes uint8 [rows, K/2], E4M3 scales uint8 [rows, K/16])."""
    w = _c(w, np.float32)
    rows, K = w.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    scales = np.zeros((rows, K // 16), np.uint8)
    lib().oracle_quantize_nvfp4(_p(w), rows, K, float(gs), _p(codes), _p(scales))
    return codes, scales


def quantize_nvfp4_bf16(x_bits, gs: float):
    """bf16 bits uint16 [rows, K] -> (E2M1 codes uint8 [rows, K], one per element; E4M3 scales uint8 [rows, K/16])."""
    x = _c(x_bits, np.uint16)
    rows, K = x.shape
    codes = np.zeros((rows, K), np.uint8)
    scales = np.zeros((rows, K // 16), np.uint8)
    lib().oracle_quantize_nvfp4_bf16(_p(x), rows, K, float(gs), _p(codes), _p(scales))
    return codes, scales


def forward_nvfp4(x_bits, ids, w, wmap, w1, w1s, w1gs, w2, w2s, w2gs, *, x_gscale: float, h_gscale: float, H: int,
                  I: int, E_global: int, E_local: int, expert_offset: int, num_shared: int, tokens=None,
                  want_act: bool = False, want_xq: bool = False, activation: int = ACT_SWIGLU, act_params=(0.0, 0.0),
                  want_y: bool = False):
    """Layer forward of the NVFP4 variant for ``tokens``: as ``forward`` with
    NVFP4 weights (w1 / w2 packed codes, E4M3 scales per 16, fp32 global scales
    w1gs / w2gs per compact expert) and NVFP4 activations (global scales
    x_gscale for x, h_gscale for the intermediate).  act_sf / xq_sf hold one
    E4M3 scale per 16 elements."""
    x = _c(x_bits, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    T, kp = ids.shape
    toks = _c(np.arange(T) if tokens is None else tokens, np.int32)
    n = toks.size
    out = np.zeros((n, H), np.float64)
    outb = np.zeros((n, H), np.uint16)
    act = np.zeros((n, kp, I), np.uint8) if want_act else None
    acts = np.zeros((n, kp, I // 16), np.uint8) if want_act else None
    xq = np.zeros((n, H), np.uint8) if want_xq else None
    xqs = np.zeros((n, H // 16), np.uint8) if want_xq else None
    ys = np.zeros((n, kp, H), np.float64) if want_y else None
    a1, s1, a2, s2 = (_c(a, np.uint8) for a in (w1, w1s, w2, w2s))
    g1, g2 = _c(w1gs, np.float32), _c(w2gs, np.float32)
    wm = _c(wmap, np.int32)
    c = (list(act_params) + [0.0, 0.0])[:2]
    rc = lib().oracle_forward_nvfp4(T, H, I, kp, E_global, E_local, expert_offset, num_shared, _p(x), _p(ids), _p(w),
                                    _p(wm), _p(a1), _p(s1), _p(g1), _p(a2), _p(s2), _p(g2), float(x_gscale),
                                    float(h_gscale), n, _p(toks), _p(out), _p(outb), _p(act), _p(acts), _p(xq),
                                    _p(xqs), int(activation), float(c[0]), float(c[1]), _p(ys))
    if rc != 0:
        raise ValueError("oracle_forward_nvfp4: a routed expert has no weights in wmap")
    res = dict(out_f64=out, out_bf16=outb)
    if want_act:
        res.update(act=act, act_sf=acts)
    if want_xq:
        res.update(xq=xq, xq_sf=xqs)
    if want_y:
        res.update(y_slot=ys)
    return res
