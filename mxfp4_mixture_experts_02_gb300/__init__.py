"""GB300 (sm_103a) fused MXFP4 Mixture-of-Experts layer forward.

A thin ctypes binding over the C ABI in ``include/moe_api.h`` (library
``_build/libmoe_gb300.so``).  The functions keep the C names; they marshal
torch tensors (device pointers) and the current CUDA stream, nothing more:
every step of the layer runs in the library's kernels.  There is no CPU or
eager fallback -- without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

from . import build as _build

__all__ = [
    "MoeShape", "MoeWeights", "MoeError", "lib", "moe_is_supported", "moe_workspace_bytes",
    "moe_quantize_mxfp4", "moe_packed_weight_bytes", "moe_pack_weights", "moe_route", "moe_sort", "moe_forward",
    "moe_layer", "moe_router", "moe_layer_router", "moe_layer_host", "moe_layer_events", "moe_layer_noalloc", "moe_get_views", "moe_get_status",
    "moe_num_sms", "moe_layer_launch_count", "quantize_expert_weights", "moe_noalloc_get_status",
    "moe_test_set_stall", "moe_set_gemm2_path", "GEMM2_AUTO", "GEMM2_SPLIT", "GEMM2_DENSE",
    "MoeNvfp4", "moe_quantize_nvfp4", "moe_pack_weights_nvfp4", "moe_layer_nvfp4", "moe_layer_nvfp4_events",
    "quantize_expert_weights_nvfp4",
    "workspace", "MOE_OK", "MOE_ERR_TIMEOUT", "MOE_ERR_WORKSPACE",
]

MOE_OK = 0
GEMM2_AUTO, GEMM2_SPLIT, GEMM2_DENSE = 0, 1, 2  # moe_set_gemm2_path
MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_ALIGN, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = -1, -2, -3, -4, -5, -6
_ERRNAMES = {-1: "MOE_ERR_NULL", -2: "MOE_ERR_SHAPE", -3: "MOE_ERR_ALIGN", -4: "MOE_ERR_WORKSPACE",
             -5: "MOE_ERR_CUDA", -6: "MOE_ERR_TIMEOUT"}


class MoeError(RuntimeError):
    def __init__(self, fn, rc):
        super().__init__("%s returned %s (%d)" % (fn, _ERRNAMES.get(rc, "?"), rc))
        self.rc = rc


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "max_T", "E_global", "E_local", "expert_offset", "top_k",
                                               "num_shared", "hidden", "inter", "block_n", "activation")] + \
               [("shared_scale", ctypes.c_float), ("act_params", ctypes.c_float * 2)]


# FC1 epilogue activations (the MOE_ACT_* values of the C header)
ACT_SWIGLU = 0        # silu(g) * u
ACT_SWIGLU_CLAMP = 1  # silu(min(g, L)) * clamp(u, -L, L), L = act_params[0]
ACT_SITU = 2          # beta tanh(g/beta) sigmoid(g) * lb tanh(u/lb), (beta, lb) = act_params


class _Weights(ctypes.Structure):
    _fields_ = [("w1", ctypes.c_void_p), ("w1_sf", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w2_sf", ctypes.c_void_p)]


class _Views(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("header", "expert_counts", "expert_offsets", "vinfo", "a_map",
                                                "c_map", "xq", "xq_sf", "act", "act_sf", "y")] + \
               [(n, ctypes.c_int32) for n in ("max_v", "rows_alloc", "y_is_bf16", "sf_tile_bytes_x",
                                              "sf_tile_bytes_act", "x_token_order")]


@dataclasses.dataclass
class MoeShape:
    T: int
    max_T: int
    E_global: int
    E_local: int
    expert_offset: int
    top_k: int
    num_shared: int
    hidden: int
    inter: int
    block_n: int
    activation: int = 0
    shared_scale: float = 1.0
    act_params: tuple = (0.0, 0.0)

    @property
    def kp(self):
        return self.top_k + self.num_shared

    def c(self) -> _Shape:
        d = dataclasses.asdict(self)
        d["act_params"] = (ctypes.c_float * 2)(*[float(v) for v in d["act_params"]])
        return _Shape(**d)


class _Nvfp4(ctypes.Structure):
    _fields_ = [("x_gscale", ctypes.c_float), ("h_gscale", ctypes.c_float), ("w1_gscale", ctypes.c_void_p),
                ("w2_gscale", ctypes.c_void_p)]


@dataclasses.dataclass
class MoeNvfp4:
    """Global scales of the NVFP4 variant (see moe_api.h): x_gscale and
    h_gscale for the activations, w1_gscale / w2_gscale device fp32 [E_tot]."""
    x_gscale: float
    h_gscale: float
    w1_gscale: torch.Tensor
    w2_gscale: torch.Tensor

    def c(self) -> _Nvfp4:
        return _Nvfp4(float(self.x_gscale), float(self.h_gscale), self.w1_gscale.data_ptr(),
                      self.w2_gscale.data_ptr())


@dataclasses.dataclass
class MoeWeights:
    """Packed expert weights (device tensors, uint8)."""
    w1: torch.Tensor
    w1_sf: torch.Tensor
    w2: torch.Tensor
    w2_sf: torch.Tensor

    def c(self) -> _Weights:
        return _Weights(self.w1.data_ptr(), self.w1_sf.data_ptr(), self.w2.data_ptr(), self.w2_sf.data_ptr())


_lib = None
_SIGS = {
    "moe_is_supported": [ctypes.c_void_p],
    "moe_workspace_bytes": [ctypes.c_void_p, ctypes.c_void_p],
    "moe_quantize_mxfp4": [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                           ctypes.c_void_p],
    "moe_packed_weight_bytes": [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p],
    "moe_pack_weights": [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                         ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
    "moe_route": [ctypes.c_void_p] * 6,
    "moe_sort": [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p],
    "moe_forward": [ctypes.c_void_p] * 5 + [ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p],
    "moe_layer": [ctypes.c_void_p] * 8 + [ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p],
    "moe_router": [ctypes.c_void_p] * 5 + [ctypes.c_size_t, ctypes.c_void_p],
    "moe_layer_router": [ctypes.c_void_p] * 9 + [ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p],
    "moe_layer_host": [ctypes.c_void_p] * 6 + [ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p],
    "moe_layer_events": [ctypes.c_void_p] * 8 + [ctypes.c_size_t] + [ctypes.c_void_p] * 3,
    "moe_layer_noalloc": [ctypes.c_void_p] * 9,
    "moe_get_views": [ctypes.c_void_p] * 3,
    "moe_get_status": [ctypes.c_void_p] * 3,
    "moe_noalloc_get_status": [ctypes.c_void_p] * 2,
    "moe_test_set_stall": [ctypes.c_uint64],
    "moe_set_gemm2_path": [ctypes.c_int32],
    "moe_quantize_nvfp4": [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + [ctypes.c_void_p] * 4,
    "moe_pack_weights_nvfp4": [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                               ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
    "moe_layer_nvfp4": [ctypes.c_void_p] * 9 + [ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p],
    "moe_layer_nvfp4_events": [ctypes.c_void_p] * 9 + [ctypes.c_size_t] + [ctypes.c_void_p] * 3,
    "moe_num_sms": [ctypes.c_void_p],
    "moe_layer_launch_count": [ctypes.c_void_p, ctypes.c_void_p],
}


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True):
    """The loaded C library.  Builds it in-tree when missing (nvcc); raises if
    that is impossible -- there is no fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB) or (build_if_missing and _build.stale()):
            if not build_if_missing:
                raise ImportError("libmoe_gb300.so is not built; run __graft_entry__.build()")
            _build.build()
        L = ctypes.CDLL(_build.LIB)
        for name, argtypes in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = argtypes
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != MOE_OK:
        raise MoeError(name, rc)
    return rc


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device=None):
    return torch.cuda.current_stream(device).cuda_stream


def _check_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("expected contiguous CUDA tensors")


# ------------------------------------------------------------------ queries
def moe_is_supported(shape: MoeShape) -> bool:
    s = shape.c()
    return bool(lib().moe_is_supported(ctypes.byref(s)))


def moe_workspace_bytes(shape: MoeShape) -> int:
    s = shape.c()
    n = ctypes.c_size_t(0)
    _call("moe_workspace_bytes", ctypes.byref(s), ctypes.byref(n))
    return n.value


def moe_layer_launch_count(shape: MoeShape) -> int:
    """Kernel launches moe_layer issues for this shape."""
    n = ctypes.c_int32()
    s = shape.c()
    _call("moe_layer_launch_count", ctypes.byref(s), ctypes.byref(n))
    return n.value


def moe_num_sms() -> int:
    n = ctypes.c_int32(0)
    _call("moe_num_sms", ctypes.byref(n))
    return n.value


def workspace(shape: MoeShape, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of the right size (torch allocates, 256-byte aligned)."""
    return torch.zeros(moe_workspace_bytes(shape), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ weights
def moe_quantize_mxfp4(w: torch.Tensor):
    """fp32 [rows, K] (device) -> (E2M1 codes uint8 [rows, K/2], E8M0 uint8 [rows, K/32])."""
    _check_cuda(w)
    rows, K = w.shape
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((rows, K // 32), dtype=torch.uint8, device=w.device)
    _call("moe_quantize_mxfp4", w.data_ptr(), rows, K, codes.data_ptr(), scales.data_ptr(), _stream(w.device))
    return codes, scales


def moe_packed_weight_bytes(experts: int, N: int, K: int, pair_halves: bool):
    """(rows per block, packed code bytes, packed scale bytes) of one weight
    matrix per expert [experts, N, K] (see moe_api.h)."""
    rb = ctypes.c_int32()
    nc = ctypes.c_size_t()
    ns = ctypes.c_size_t()
    _call("moe_packed_weight_bytes", experts, N, K, 1 if pair_halves else 0, ctypes.byref(rb), ctypes.byref(nc),
          ctypes.byref(ns))
    return rb.value, nc.value, ns.value


def moe_pack_weights(codes: torch.Tensor, scales: torch.Tensor, pair_halves: bool):
    """Row-major MXFP4 of one weight matrix per expert -- codes uint8 [E, N, K/2],
    scales uint8 [E, N, K/32] -- to the tile-major layout the GEMMs stream
    (see moe_api.h).  Returns (packed_codes, packed_scales), flat uint8."""
    _check_cuda(codes, scales)
    E, N, K2 = codes.shape
    _, nc, ns = moe_packed_weight_bytes(E, N, 2 * K2, pair_halves)
    pc = torch.empty(nc, dtype=torch.uint8, device=codes.device)
    ps = torch.empty(ns, dtype=torch.uint8, device=codes.device)
    _call("moe_pack_weights", codes.data_ptr(), scales.data_ptr(), E, N, 2 * K2, 1 if pair_halves else 0,
          pc.data_ptr(), ps.data_ptr(), _stream(codes.device))
    return pc, ps


def quantize_expert_weights(w1: torch.Tensor, w2: torch.Tensor, keep_rowmajor: bool = False):
    """fp32 W1 [E, 2I, H] and W2 [E, H, I] (device) -> packed MoeWeights (and, if
    asked, the row-major codes and scales (c1, s1, c2, s2) for inspection)."""
    E, I2, H = w1.shape
    I = w2.shape[2]
    c1, s1 = moe_quantize_mxfp4(w1.reshape(E * I2, H))
    c2, s2 = moe_quantize_mxfp4(w2.reshape(E * H, I))
    c1, s1 = c1.reshape(E, I2, H // 2), s1.reshape(E, I2, H // 32)
    c2, s2 = c2.reshape(E, H, I // 2), s2.reshape(E, H, I // 32)
    p1, q1 = moe_pack_weights(c1, s1, True)
    p2, q2 = moe_pack_weights(c2, s2, False)
    wts = MoeWeights(p1, q1, p2, q2)
    if keep_rowmajor:
        return wts, (c1, s1, c2, s2)
    return wts


def moe_quantize_nvfp4(w: torch.Tensor):
    """fp32 [experts, rows, K] (device) -> (gscale fp32 [experts], E2M1 codes uint8
    [experts, rows, K/2], E4M3 scales uint8 [experts, rows, K/16])."""
    _check_cuda(w)
    E, rows, K = w.shape
    gs = torch.empty(E, dtype=torch.float32, device=w.device)
    codes = torch.empty((E, rows, K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((E, rows, K // 16), dtype=torch.uint8, device=w.device)
    _call("moe_quantize_nvfp4", w.data_ptr(), E, rows, K, gs.data_ptr(), codes.data_ptr(), scales.data_ptr(),
          _stream(w.device))
    return gs, codes, scales


def moe_pack_weights_nvfp4(codes: torch.Tensor, scales: torch.Tensor, pair_halves: bool):
    """NVFP4 codes uint8 [E, N, K/2] and scales uint8 [E, N, K/16] to the
    tile-major layout (see moe_api.h).  Returns (packed_codes, packed_scales), flat uint8."""
    _check_cuda(codes, scales)
    E, N, K2 = codes.shape
    pc = torch.empty(E * N * K2, dtype=torch.uint8, device=codes.device)
    ps = torch.empty(E * N * (2 * K2 // 16), dtype=torch.uint8, device=codes.device)
    _call("moe_pack_weights_nvfp4", codes.data_ptr(), scales.data_ptr(), E, N, 2 * K2, 1 if pair_halves else 0,
          pc.data_ptr(), ps.data_ptr(), _stream(codes.device))
    return pc, ps


def quantize_expert_weights_nvfp4(w1: torch.Tensor, w2: torch.Tensor, x_gscale: float, h_gscale: float,
                                  keep_rowmajor: bool = False):
    """fp32 W1 [E, 2I, H] and W2 [E, H, I] (device) -> (packed MoeWeights, MoeNvfp4)
    (and, if asked, the row-major (c1, s1, c2, s2))."""
    g1, c1, s1 = moe_quantize_nvfp4(w1)
    g2, c2, s2 = moe_quantize_nvfp4(w2)
    p1, q1 = moe_pack_weights_nvfp4(c1, s1, True)
    p2, q2 = moe_pack_weights_nvfp4(c2, s2, False)
    res = (MoeWeights(p1, q1, p2, q2), MoeNvfp4(x_gscale, h_gscale, g1, g2))
    if keep_rowmajor:
        return res + ((c1, s1, c2, s2),)
    return res


# ------------------------------------------------------------------ the layer
def moe_route(shape: MoeShape, logits, shared_logit=None, topk_ids=None, topk_w=None):
    _check_cuda(logits, shared_logit)
    T = shape.T
    if topk_ids is None:
        topk_ids = torch.empty((T, shape.kp), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, shape.kp), dtype=torch.float32, device=logits.device)
    s = shape.c()
    _call("moe_route", ctypes.byref(s), logits.data_ptr(), _ptr(shared_logit), topk_ids.data_ptr(),
          topk_w.data_ptr(), _stream(logits.device))
    return topk_ids, topk_w


def moe_sort(shape: MoeShape, topk_ids, ws):
    _check_cuda(topk_ids, ws)
    s = shape.c()
    _call("moe_sort", ctypes.byref(s), topk_ids.data_ptr(), ws.data_ptr(), ws.numel(), _stream(ws.device))


def moe_forward(shape: MoeShape, x, weights: MoeWeights, topk_w, ws, out=None):
    _check_cuda(x, topk_w, ws)
    if out is None:
        out = torch.empty((shape.T, shape.hidden), dtype=torch.bfloat16, device=x.device)
    s, w = shape.c(), weights.c()
    _call("moe_forward", ctypes.byref(s), x.data_ptr(), ctypes.byref(w), topk_w.data_ptr(), ws.data_ptr(),
          ws.numel(), out.data_ptr(), _stream(x.device))
    return out


def moe_router(shape: MoeShape, x, wr, ws, logits=None):
    """Router GEMM: bf16 x [T, H] times the bf16 router matrix wr [E_global, H] -> fp32 logits [T, E_global]."""
    _check_cuda(x, wr, ws)
    if logits is None:
        logits = torch.empty((shape.T, shape.E_global), dtype=torch.float32, device=x.device)
    s = shape.c()
    _call("moe_router", ctypes.byref(s), x.data_ptr(), wr.data_ptr(), logits.data_ptr(), ws.data_ptr(),
          ws.numel(), _stream(x.device))
    return logits


def moe_layer_router(shape: MoeShape, wr, shared_logit, x, weights: MoeWeights, ws, logits=None, topk_ids=None,
                     topk_w=None, out=None):
    """The layer from x and the router matrix: router GEMM -> route -> sort -> forward, one launch chain.
    Returns (out, logits, topk_ids, topk_w)."""
    _check_cuda(wr, shared_logit, x, ws)
    dev = x.device
    if logits is None:
        logits = torch.empty((shape.T, shape.E_global), dtype=torch.float32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((shape.T, shape.kp), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((shape.T, shape.kp), dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty((shape.T, shape.hidden), dtype=torch.bfloat16, device=dev)
    s, w = shape.c(), weights.c()
    _call("moe_layer_router", ctypes.byref(s), wr.data_ptr(), _ptr(shared_logit), x.data_ptr(), ctypes.byref(w),
          logits.data_ptr(), topk_ids.data_ptr(), topk_w.data_ptr(), ws.data_ptr(), ws.numel(), out.data_ptr(),
          _stream(dev))
    return out, logits, topk_ids, topk_w


def moe_layer(shape: MoeShape, logits, shared_logit, x, weights: MoeWeights, ws, topk_ids=None, topk_w=None,
              out=None):
    _check_cuda(logits, shared_logit, x, ws)
    dev = x.device
    if topk_ids is None:
        topk_ids = torch.empty((shape.T, shape.kp), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((shape.T, shape.kp), dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty((shape.T, shape.hidden), dtype=torch.bfloat16, device=dev)
    s, w = shape.c(), weights.c()
    _call("moe_layer", ctypes.byref(s), logits.data_ptr(), _ptr(shared_logit), x.data_ptr(), ctypes.byref(w),
          topk_ids.data_ptr(), topk_w.data_ptr(), ws.data_ptr(), ws.numel(), out.data_ptr(), _stream(dev))
    return out, topk_ids, topk_w


def moe_layer_nvfp4(shape: MoeShape, nv: MoeNvfp4, logits, shared_logit, x, weights: MoeWeights, ws,
                    topk_ids=None, topk_w=None, out=None):
    """moe_layer in the NVFP4 variant (128-row tiles)."""
    _check_cuda(logits, shared_logit, x, ws)
    dev = x.device
    if topk_ids is None:
        topk_ids = torch.empty((shape.T, shape.kp), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((shape.T, shape.kp), dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty((shape.T, shape.hidden), dtype=torch.bfloat16, device=dev)
    s, w, n = shape.c(), weights.c(), nv.c()
    _call("moe_layer_nvfp4", ctypes.byref(s), ctypes.byref(n), logits.data_ptr(), _ptr(shared_logit), x.data_ptr(),
          ctypes.byref(w), topk_ids.data_ptr(), topk_w.data_ptr(), ws.data_ptr(), ws.numel(), out.data_ptr(),
          _stream(dev))
    return out, topk_ids, topk_w


def moe_layer_nvfp4_events(shape: MoeShape, nv: MoeNvfp4, logits, shared_logit, x, weights: MoeWeights, ws, topk_ids,
                           topk_w, out, events):
    """moe_layer_nvfp4 with the 7 stage events of moe_layer_events."""
    _check_cuda(logits, shared_logit, x, ws)
    stream = torch.cuda.current_stream(x.device)
    for ev in events:
        if not ev.cuda_event:
            ev.record(stream)
    arr = (ctypes.c_void_p * 7)(*[ev.cuda_event for ev in events])
    s, w, n = shape.c(), weights.c(), nv.c()
    _call("moe_layer_nvfp4_events", ctypes.byref(s), ctypes.byref(n), logits.data_ptr(), _ptr(shared_logit),
          x.data_ptr(), ctypes.byref(w), topk_ids.data_ptr(), topk_w.data_ptr(), ws.data_ptr(), ws.numel(),
          out.data_ptr(), arr, _stream(x.device))
    return out


def moe_layer_events(shape: MoeShape, logits, shared_logit, x, weights: MoeWeights, ws, topk_ids, topk_w, out,
                     events):
    """moe_layer with 7 torch.cuda.Events recorded at the stage boundaries
    (before route, after route / sort / gather / FC1 / FC2 / combine)."""
    _check_cuda(logits, shared_logit, x, ws)
    stream = torch.cuda.current_stream(x.device)
    for ev in events:
        if not ev.cuda_event:  # torch creates the CUDA event on its first record
            ev.record(stream)
    arr = (ctypes.c_void_p * 7)(*[ev.cuda_event for ev in events])
    s, w = shape.c(), weights.c()
    _call("moe_layer_events", ctypes.byref(s), logits.data_ptr(), _ptr(shared_logit), x.data_ptr(), ctypes.byref(w),
          topk_ids.data_ptr(), topk_w.data_ptr(), ws.data_ptr(), ws.numel(), out.data_ptr(), arr,
          _stream(x.device))
    return out


def moe_layer_noalloc(shape: MoeShape, logits, shared_logit, x, weights: MoeWeights, topk_ids=None, topk_w=None,
                      out=None):
    """moe_layer without a workspace argument, for callers that cannot
    allocate device memory: the scratch is the library's fixed 32 MiB device
    array (shapes needing more raise MoeError(MOE_ERR_WORKSPACE)).  Calls that
    run concurrently on the GPU share that array and must be serialised."""
    _check_cuda(logits, shared_logit, x)
    dev = x.device
    if topk_ids is None:
        topk_ids = torch.empty((shape.T, shape.kp), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((shape.T, shape.kp), dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty((shape.T, shape.hidden), dtype=torch.bfloat16, device=dev)
    s, w = shape.c(), weights.c()
    _call("moe_layer_noalloc", ctypes.byref(s), logits.data_ptr(), _ptr(shared_logit), x.data_ptr(),
          ctypes.byref(w), topk_ids.data_ptr(), topk_w.data_ptr(), out.data_ptr(), _stream(dev))
    return out, topk_ids, topk_w


def moe_layer_host(shape: MoeShape, logits_h, shared_logit_h, x_h, weights: MoeWeights, ws, out_h):
    """Host tensors in and out (pinned CPU tensors recommended); asynchronous on
    the current stream -- synchronise before reading out_h."""
    s, w = shape.c(), weights.c()
    _call("moe_layer_host", ctypes.byref(s), logits_h.data_ptr(), _ptr(shared_logit_h), x_h.data_ptr(),
          ctypes.byref(w), ws.data_ptr(), ws.numel(), out_h.data_ptr(), _stream(ws.device))
    return out_h


def moe_get_status(ws):
    st, det = ctypes.c_int32(0), ctypes.c_int32(0)
    _call("moe_get_status", ws.data_ptr(), ctypes.byref(st), ctypes.byref(det))
    return st.value, det.value


def moe_noalloc_get_status():
    """Status word of moe_layer_noalloc's scratch array on the current device (synchronous)."""
    st, det = ctypes.c_int32(0), ctypes.c_int32(0)
    _call("moe_noalloc_get_status", ctypes.byref(st), ctypes.byref(det))
    return st.value, det.value


def moe_set_gemm2_path(path: int):
    """Force the GEMM2 path of later calls: GEMM2_AUTO (the device gate's rule),
    GEMM2_SPLIT or GEMM2_DENSE (see moe_api.h)."""
    _call("moe_set_gemm2_path", int(path))


def moe_test_set_stall(stall_ns: int):
    """Test hook: while nonzero, every FC1 launch stalls its MMA thread on a
    barrier nothing arrives on for stall_ns, so the call reports
    MOE_ERR_TIMEOUT (site 5) in its status word.  0 turns it off."""
    _call("moe_test_set_stall", int(stall_ns))


def moe_get_views(shape: MoeShape, ws):
    """Workspace views as torch tensors (sharing the workspace memory)."""
    s = shape.c()
    v = _Views()
    _call("moe_get_views", ctypes.byref(s), ws.data_ptr(), ctypes.byref(v))
    base = ws.data_ptr()

    def sub(ptr, nbytes, dtype):
        off = ptr - base
        return ws[off:off + nbytes].view(dtype)

    Et = shape.E_local + shape.num_shared
    hdr = sub(v.header, 64 * 4, torch.int32)
    R_max = shape.max_T * shape.kp
    return dict(
        header=hdr, expert_counts=sub(v.expert_counts, Et * 4, torch.int32),
        expert_offsets=sub(v.expert_offsets, (Et + 1) * 4, torch.int32),
        vinfo=sub(v.vinfo, v.max_v * 16, torch.int32).view(v.max_v, 4),
        a_map=sub(v.a_map, R_max * 4, torch.int32), c_map=sub(v.c_map, R_max * 4, torch.int32),
        xq=(sub(v.xq, shape.max_T * shape.hidden, torch.uint8).view(shape.max_T, shape.hidden) if v.x_token_order
            else sub(v.xq, v.rows_alloc * shape.hidden, torch.uint8).view(v.rows_alloc, shape.hidden)),
        xq_sf=(sub(v.xq_sf, shape.max_T * (shape.hidden // 32), torch.uint8).view(shape.max_T, shape.hidden // 32)
               if v.x_token_order
               else sub(v.xq_sf, v.max_v * v.sf_tile_bytes_x, torch.uint8).view(v.max_v, v.sf_tile_bytes_x)),
        x_token_order=v.x_token_order,
        act=sub(v.act, v.rows_alloc * shape.inter, torch.uint8).view(v.rows_alloc, shape.inter),
        act_sf=sub(v.act_sf, v.max_v * v.sf_tile_bytes_act, torch.uint8).view(v.max_v, v.sf_tile_bytes_act),
        y=(sub(v.y, R_max * shape.hidden * 2, torch.bfloat16) if v.y_is_bf16
           else sub(v.y, R_max * shape.hidden * 4, torch.float32)).view(R_max, shape.hidden),
        max_v=v.max_v, rows_alloc=v.rows_alloc, y_is_bf16=v.y_is_bf16,
    )
