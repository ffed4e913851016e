"""Seeded synthetic inputs for the MXFP4 MoE layer (see ``synth.h``).

The generator is one counter hash compiled twice: ``synth_host.c`` for host
arrays (the oracle's inputs) and ``synth_cuda.cu`` for device arrays (full-size
inputs straight into HBM).  Both produce identical bits.  Nothing here
quantises, routes or multiplies: those steps belong to the oracle and to the
GPU library, each on its own.

Workload recipe (the layer's five configurations; sigma is a standard deviation):
  x            bf16 ~ N(0, 1)                              (stream 1)
  logits       fp32 ~ N(0, 1) (+ Zipf popularity bias)     (stream 2)
               tiny config: fp32(x @ Wr) with Wr fp32 ~ N(0, 0.05) [H, E] (stream 3)
  W1, W2       fp32 ~ N(0, 0.02), per global expert id      (streams 4, 5)
  shared logit bf16 ~ N(0, 1)                              (stream 6)
N(0, 1) is the exact Irwin-Hall(12) - 6 approximation described in synth.h.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_HOST_SO = os.path.join(_BUILD, "libsynth_host.so")
_CUDA_SO = os.path.join(_BUILD, "libsynth_cuda.so")
_host = None
_cuda = None

STREAM_X, STREAM_LOGITS, STREAM_ROUTER, STREAM_W1, STREAM_W2, STREAM_SHARED = 1, 2, 3, 4, 5, 6


# ------------------------------------------------------------------ configs
@dataclasses.dataclass(frozen=True)
class MoeConfig:
    name: str
    seed: int
    T: int
    E_global: int
    E_local: int
    expert_offset: int
    top_k: int
    num_shared: int
    hidden: int
    inter: int
    block_n: int
    router: str = "normal"          # "normal": logits ~ N(0,1); "matrix": fp32(x @ Wr)
    router_sigma: float = 0.05
    zipf_s: float = 0.0             # > 0: logits += -s * ln(e + 1)
    shared_scale: float = 1.0
    weight_sigma: float = 0.02
    activation: int = 0             # FC1 activation: 0 SwiGLU, 1 clamped SwiGLU, 2 SiTU
    act_params: tuple = (0.0, 0.0)  # (limit,) or (beta, linear beta)

    @property
    def kp(self) -> int:
        return self.top_k + self.num_shared

    @property
    def global_ids(self):
        """Global ids of the local weight slots: the routed slice, then shared."""
        ids = list(range(self.expert_offset, self.expert_offset + self.E_local))
        ids += [self.E_global + s for s in range(self.num_shared)]
        return np.asarray(ids, np.int64)

    def replace(self, **kw) -> "MoeConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": MoeConfig("tiny", 0, T=4, E_global=8, E_local=8, expert_offset=0, top_k=2, num_shared=0,
                      hidden=512, inter=128, block_n=16, router="matrix"),
    "decode_t32": MoeConfig("decode_t32", 1, T=32, E_global=896, E_local=896, expert_offset=0, top_k=16,
                            num_shared=0, hidden=3584, inter=384, block_n=32),
    "ep_slice_t64": MoeConfig("ep_slice_t64", 2, T=64, E_global=896, E_local=448, expert_offset=448, top_k=16,
                              num_shared=0, hidden=3584, inter=384, block_n=16),
    "skewed_shared_t256": MoeConfig("skewed_shared_t256", 3, T=256, E_global=896, E_local=896, expert_offset=0,
                                    top_k=16, num_shared=1, hidden=3584, inter=384, block_n=32, zipf_s=1.1),
    "prefill_t32768": MoeConfig("prefill_t32768", 4, T=32768, E_global=896, E_local=896, expert_offset=0,
                                top_k=16, num_shared=0, hidden=3584, inter=384, block_n=128),
}
CONFIG_ORDER = ["tiny", "decode_t32", "ep_slice_t64", "skewed_shared_t256", "prefill_t32768"]


def logit_bias(cfg: MoeConfig):
    """Zipf(s) popularity bias over expert ids: log-pmf up to a constant."""
    if cfg.zipf_s <= 0:
        return None
    return np.asarray([-cfg.zipf_s * math.log(e + 1.0) for e in range(cfg.E_global)], np.float64)


# ------------------------------------------------------------------ building
def _stale(so, srcs):
    return not os.path.exists(so) or any(os.path.getmtime(s) > os.path.getmtime(so) for s in srcs)


def build_host(force: bool = False) -> str:
    src = os.path.join(_HERE, "synth_host.c")
    if force or _stale(_HOST_SO, [src, os.path.join(_HERE, "synth.h")]):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _HOST_SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, src])
        os.replace(tmp, _HOST_SO)
    return _HOST_SO


def build_cuda(force: bool = False) -> str:
    src = os.path.join(_HERE, "synth_cuda.cu")
    if force or _stale(_CUDA_SO, [src, os.path.join(_HERE, "synth.h")]):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _CUDA_SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               "-fmad=false", "-shared", "-Xcompiler", "-fPIC", "-o", tmp, src])
        os.replace(tmp, _CUDA_SO)
    return _CUDA_SO


def host_lib():
    global _host
    if _host is None:
        build_host()
        L = ctypes.CDLL(_HOST_SO)
        u64, i64, P, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        L.synth_x.argtypes = [u64, i64, i64, i64, P]
        L.synth_logits.argtypes = [u64, i64, i64, i64, P, P]
        L.synth_router.argtypes = [u64, i64, i64, dbl, P]
        L.synth_shared_logit.argtypes = [u64, i64, i64, P]
        L.synth_w1.argtypes = [u64, i64, i64, P, i64, dbl, P]
        L.synth_w2.argtypes = [u64, i64, i64, P, i64, dbl, P]
        L.synth_normal_q16_range.argtypes = [u64, u64, u64, i64, P]
        for f in (L.synth_x, L.synth_logits, L.synth_router, L.synth_shared_logit, L.synth_w1, L.synth_w2,
                  L.synth_normal_q16_range):
            f.restype = None
        _host = L
    return _host


def cuda_lib():
    global _cuda
    if _cuda is None:
        build_cuda()
        L = ctypes.CDLL(_CUDA_SO)
        u64, i64, P, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        L.synth_x_cuda.argtypes = [u64, i64, i64, i64, P, P]
        L.synth_logits_cuda.argtypes = [u64, i64, i64, i64, P, P, P]
        L.synth_shared_logit_cuda.argtypes = [u64, i64, i64, P, P]
        L.synth_w1_cuda.argtypes = [u64, i64, i64, P, i64, dbl, P, P]
        L.synth_w2_cuda.argtypes = [u64, i64, i64, P, i64, dbl, P, P]
        L.synth_normal_q16_range_cuda.argtypes = [u64, u64, u64, i64, P, P]
        for f in (L.synth_x_cuda, L.synth_logits_cuda, L.synth_shared_logit_cuda, L.synth_w1_cuda,
                  L.synth_w2_cuda, L.synth_normal_q16_range_cuda):
            f.restype = ctypes.c_int
        _cuda = L
    return _cuda


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ host arrays
def x_host(cfg: MoeConfig, t0: int = 0, T: int | None = None):
    T = cfg.T if T is None else T
    out = np.zeros((T, cfg.hidden), np.uint16)
    host_lib().synth_x(cfg.seed, t0, T, cfg.hidden, _p(out))
    return out


def router_host(cfg: MoeConfig):
    out = np.zeros((cfg.hidden, cfg.E_global), np.float32)
    host_lib().synth_router(cfg.seed, cfg.hidden, cfg.E_global, cfg.router_sigma, _p(out))
    return out


def bf16_bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def logits_host(cfg: MoeConfig, t0: int = 0, T: int | None = None):
    """fp32 [T, Eg].  'matrix' router: fp32(sum_h fp64(x) fp64(Wr)), computed here once."""
    T = cfg.T if T is None else T
    if cfg.router == "matrix":
        # Products bf16 * fp32 are exact in fp64; fsum rounds their sum once,
        # so the logits do not depend on the host's BLAS summation order.
        x = bf16_bits_to_f64(x_host(cfg, t0, T))
        wr = router_host(cfg).astype(np.float64)
        out = np.empty((T, cfg.E_global), np.float32)
        for t in range(T):
            for e in range(cfg.E_global):
                out[t, e] = np.float32(math.fsum(x[t] * wr[:, e]))
        return out
    out = np.zeros((T, cfg.E_global), np.float32)
    bias = logit_bias(cfg)
    host_lib().synth_logits(cfg.seed, t0, T, cfg.E_global, _p(bias), _p(out))
    return out


def shared_logit_host(cfg: MoeConfig, t0: int = 0, T: int | None = None):
    T = cfg.T if T is None else T
    out = np.zeros(T * cfg.num_shared, np.uint16)
    if cfg.num_shared:
        host_lib().synth_shared_logit(cfg.seed, t0, T, _p(out))
    return out.reshape(T, cfg.num_shared)


def w1_host(cfg: MoeConfig, global_ids):
    g = np.ascontiguousarray(global_ids, np.int64)
    out = np.zeros((g.size, 2 * cfg.inter, cfg.hidden), np.float32)
    host_lib().synth_w1(cfg.seed, cfg.hidden, cfg.inter, _p(g), g.size, cfg.weight_sigma, _p(out))
    return out


def w2_host(cfg: MoeConfig, global_ids):
    g = np.ascontiguousarray(global_ids, np.int64)
    out = np.zeros((g.size, cfg.hidden, cfg.inter), np.float32)
    host_lib().synth_w2(cfg.seed, cfg.hidden, cfg.inter, _p(g), g.size, cfg.weight_sigma, _p(out))
    return out


def normal_q16_host(seed: int, stream: int, i0: int, n: int):
    out = np.zeros(n, np.int32)
    host_lib().synth_normal_q16_range(seed, stream, i0, n, _p(out))
    return out


# ------------------------------------------------------------------ device tensors
def _check(rc, what):
    if rc != 0:
        raise RuntimeError("%s failed: cudaError %d" % (what, rc))


def x_device(cfg: MoeConfig, device="cuda", t0: int = 0, T: int | None = None):
    import torch
    T = cfg.T if T is None else T
    out = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device=device)
    s = torch.cuda.current_stream(out.device).cuda_stream
    _check(cuda_lib().synth_x_cuda(cfg.seed, t0, T, cfg.hidden, out.data_ptr(), s), "synth_x_cuda")
    return out


def logits_device(cfg: MoeConfig, device="cuda", t0: int = 0, T: int | None = None):
    import torch
    T = cfg.T if T is None else T
    if cfg.router == "matrix":
        return torch.from_numpy(logits_host(cfg, t0, T)).to(device)
    out = torch.empty((T, cfg.E_global), dtype=torch.float32, device=device)
    bias = logit_bias(cfg)
    bias_d = None if bias is None else torch.from_numpy(bias).to(device)
    s = torch.cuda.current_stream(out.device).cuda_stream
    _check(cuda_lib().synth_logits_cuda(cfg.seed, t0, T, cfg.E_global,
                                        None if bias_d is None else bias_d.data_ptr(), out.data_ptr(), s),
           "synth_logits_cuda")
    torch.cuda.current_stream(out.device).synchronize()
    return out


def shared_logit_device(cfg: MoeConfig, device="cuda", t0: int = 0, T: int | None = None):
    import torch
    T = cfg.T if T is None else T
    out = torch.empty((T, max(cfg.num_shared, 1)), dtype=torch.bfloat16, device=device)
    if cfg.num_shared:
        s = torch.cuda.current_stream(out.device).cuda_stream
        _check(cuda_lib().synth_shared_logit_cuda(cfg.seed, t0, T, out.data_ptr(), s), "synth_shared_logit_cuda")
    return out[:, :cfg.num_shared]


def w1_device(cfg: MoeConfig, global_ids, device="cuda"):
    import torch
    g = torch.as_tensor(np.ascontiguousarray(global_ids, np.int64)).to(device)
    out = torch.empty((g.numel(), 2 * cfg.inter, cfg.hidden), dtype=torch.float32, device=device)
    s = torch.cuda.current_stream(out.device).cuda_stream
    _check(cuda_lib().synth_w1_cuda(cfg.seed, cfg.hidden, cfg.inter, g.data_ptr(), g.numel(), cfg.weight_sigma,
                                    out.data_ptr(), s), "synth_w1_cuda")
    torch.cuda.current_stream(out.device).synchronize()
    return out


def w2_device(cfg: MoeConfig, global_ids, device="cuda"):
    import torch
    g = torch.as_tensor(np.ascontiguousarray(global_ids, np.int64)).to(device)
    out = torch.empty((g.numel(), cfg.hidden, cfg.inter), dtype=torch.float32, device=device)
    s = torch.cuda.current_stream(out.device).cuda_stream
    _check(cuda_lib().synth_w2_cuda(cfg.seed, cfg.hidden, cfg.inter, g.data_ptr(), g.numel(), cfg.weight_sigma,
                                    out.data_ptr(), s), "synth_w2_cuda")
    torch.cuda.current_stream(out.device).synchronize()
    return out


def normal_q16_device(seed: int, stream: int, i0: int, n: int, device="cuda"):
    import torch
    out = torch.empty(n, dtype=torch.int32, device=device)
    s = torch.cuda.current_stream(out.device).cuda_stream
    _check(cuda_lib().synth_normal_q16_range_cuda(seed, stream, i0, n, out.data_ptr(), s), "synth_normal_q16")
    torch.cuda.current_stream(out.device).synchronize()
    return out
