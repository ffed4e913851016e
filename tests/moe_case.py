"""Builds MoE layer test cases: device inputs for the GPU library and, for the
tokens being checked, the oracle's own independent computation.

GPU side : x / logits / shared logit / fp32 weights from the CUDA build of the
           seeded generator; weights quantised by the library
           (moe_quantize_mxfp4 + moe_pack_weights).
Oracle   : the same seeded inputs from the host build of the generator;
           routing, sort, weight quantisation and forward by the oracle.
Nothing computed by the GPU library feeds the oracle.
"""
from __future__ import annotations

import concurrent.futures
import os

import numpy as np
import torch

import mxfp4_mixture_experts_02_gb300 as moe
import oracle
import synth


def shape_of(cfg: synth.MoeConfig, T: int | None = None) -> moe.MoeShape:
    T = cfg.T if T is None else T
    return moe.MoeShape(T=T, max_T=max(T, 1), E_global=cfg.E_global, E_local=cfg.E_local,
                        expert_offset=cfg.expert_offset, top_k=cfg.top_k, num_shared=cfg.num_shared,
                        hidden=cfg.hidden, inter=cfg.inter, block_n=cfg.block_n, shared_scale=cfg.shared_scale,
                        activation=cfg.activation, act_params=tuple(cfg.act_params))


def device_weights(cfg: synth.MoeConfig, chunk: int = 64, keep_rowmajor: bool = False):
    """Packed weights of all local experts (+shared), generated and quantised
    on the device chunk by chunk, packed by the library."""
    gids = cfg.global_ids
    E, H, I = gids.size, cfg.hidden, cfg.inter
    dev = "cuda"
    c1 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=dev)
    c2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=dev)
    s1 = torch.empty((E, 2 * I, H // 32), dtype=torch.uint8, device=dev)
    s2 = torch.empty((E, H, I // 32), dtype=torch.uint8, device=dev)
    for c0 in range(0, E, chunk):
        ids = gids[c0:c0 + chunk]
        n = ids.size
        c, s = moe.moe_quantize_mxfp4(synth.w1_device(cfg, ids).reshape(n * 2 * I, H))
        c1[c0:c0 + n] = c.reshape(n, 2 * I, H // 2)
        s1[c0:c0 + n] = s.reshape(n, 2 * I, H // 32)
        c, s = moe.moe_quantize_mxfp4(synth.w2_device(cfg, ids).reshape(n * H, I))
        c2[c0:c0 + n] = c.reshape(n, H, I // 2)
        s2[c0:c0 + n] = s.reshape(n, H, I // 32)
    p1, q1 = moe.moe_pack_weights(c1, s1, True)
    p2, q2 = moe.moe_pack_weights(c2, s2, False)
    wts = moe.MoeWeights(p1, q1, p2, q2)
    torch.cuda.synchronize()
    if keep_rowmajor:
        return wts, (c1, s1, c2, s2)
    del c1, c2, s1, s2
    torch.cuda.empty_cache()
    return wts


def device_weights_nvfp4(cfg: synth.MoeConfig, x_gscale: float, h_gscale: float, chunk: int = 64):
    """NVFP4 weights of all local experts (+shared), generated on the device,
    quantised (per-expert global scales) and packed by the library:
    (MoeWeights, MoeNvfp4)."""
    gids = cfg.global_ids
    E, H, I = gids.size, cfg.hidden, cfg.inter
    dev = "cuda"
    c1 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=dev)
    c2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=dev)
    s1 = torch.empty((E, 2 * I, H // 16), dtype=torch.uint8, device=dev)
    s2 = torch.empty((E, H, I // 16), dtype=torch.uint8, device=dev)
    g1 = torch.empty(E, dtype=torch.float32, device=dev)
    g2 = torch.empty(E, dtype=torch.float32, device=dev)
    for c0 in range(0, E, chunk):
        ids = gids[c0:c0 + chunk]
        n = ids.size
        g1[c0:c0 + n], c1[c0:c0 + n], s1[c0:c0 + n] = moe.moe_quantize_nvfp4(synth.w1_device(cfg, ids))
        g2[c0:c0 + n], c2[c0:c0 + n], s2[c0:c0 + n] = moe.moe_quantize_nvfp4(synth.w2_device(cfg, ids))
    p1, q1 = moe.moe_pack_weights_nvfp4(c1, s1, True)
    p2, q2 = moe.moe_pack_weights_nvfp4(c2, s2, False)
    torch.cuda.synchronize()
    del c1, c2, s1, s2
    torch.cuda.empty_cache()
    return moe.MoeWeights(p1, q1, p2, q2), moe.MoeNvfp4(x_gscale, h_gscale, g1, g2)


def device_inputs(cfg: synth.MoeConfig, T: int | None = None):
    T = cfg.T if T is None else T
    x = synth.x_device(cfg, T=T)
    logits = synth.logits_device(cfg, T=T)
    sl = synth.shared_logit_device(cfg, T=T).contiguous() if cfg.num_shared else None
    return x, logits, sl


# Oracle-quantised expert weights, shared by the cases of one weight set
# (seed and shapes); one set per format is held at a time.
_ORACLE_WEIGHTS = {}


def _shared_weight_cache(cfg, kind):
    key = (cfg.seed, cfg.E_global, cfg.E_local, cfg.expert_offset, cfg.num_shared, cfg.hidden, cfg.inter)
    held = _ORACLE_WEIGHTS.get(kind)
    if held is None or held[0] != key:
        held = _ORACLE_WEIGHTS[kind] = (key, {})
    return held[1]


class OracleCase:
    """The oracle's computation of a config for a subset of tokens."""

    def __init__(self, cfg: synth.MoeConfig, T: int | None = None, logits=None):
        self.cfg = cfg
        self.T = cfg.T if T is None else T
        self.x = synth.x_host(cfg, T=self.T)
        # logits: the oracle's own router logits when the layer starts from the router matrix
        self.logits = synth.logits_host(cfg, T=self.T) if logits is None else logits
        self.shared = synth.shared_logit_host(cfg, T=self.T)
        self.ids, self.w = oracle.route(self.logits, cfg.top_k, cfg.num_shared, self.shared, cfg.shared_scale)
        self.sort = oracle.sort(self.ids, cfg.E_global, cfg.E_local, cfg.expert_offset, cfg.num_shared, cfg.block_n)
        self._wcache = _shared_weight_cache(cfg, "mxfp4")

    def local_of(self, gid):
        c = self.cfg
        if gid >= c.E_global:
            return c.E_local + gid - c.E_global
        if c.expert_offset <= gid < c.expert_offset + c.E_local:
            return gid - c.expert_offset
        return -1

    def expert_weights(self, locals_):
        """Oracle-quantised weights of the given local experts (cached; the
        experts are generated and quantised on all host cores)."""
        c = self.cfg
        need = [e for e in locals_ if e not in self._wcache]

        def one(chunk):
            gids = c.global_ids[chunk]
            f1 = synth.w1_host(c, gids)
            f2 = synth.w2_host(c, gids)
            return [oracle.quantize_mxfp4(f1[k]) + oracle.quantize_mxfp4(f2[k]) for k in range(len(chunk))]

        if need:
            chunks = [need[i:i + 4] for i in range(0, len(need), 4)]
            with concurrent.futures.ThreadPoolExecutor(max_workers=host_threads()) as ex:
                for chunk, q in zip(chunks, ex.map(one, chunks)):
                    for e, qe in zip(chunk, q):
                        self._wcache[e] = qe
        return [self._wcache[e] for e in locals_]

    def expert_weights_nvfp4(self, locals_):
        """Oracle NVFP4 weights (codes, scales, global scale for W1 then W2) of
        the given local experts (cached; all host cores)."""
        c = self.cfg
        if "_wcache_nv" not in self.__dict__:
            self._wcache_nv = _shared_weight_cache(c, "nvfp4")
        cache = self._wcache_nv
        need = [e for e in locals_ if e not in cache]

        def one(chunk):
            gids = c.global_ids[chunk]
            f1 = synth.w1_host(c, gids)
            f2 = synth.w2_host(c, gids)
            out = []
            for k in range(len(chunk)):
                g1, g2 = oracle.nvfp4_global_scale(f1[k]), oracle.nvfp4_global_scale(f2[k])
                out.append(oracle.quantize_nvfp4(f1[k], g1) + (g1,) + oracle.quantize_nvfp4(f2[k], g2) + (g2,))
            return out

        if need:
            chunks = [need[i:i + 4] for i in range(0, len(need), 4)]
            with concurrent.futures.ThreadPoolExecutor(max_workers=host_threads()) as ex:
                for chunk, q in zip(chunks, ex.map(one, chunks)):
                    for e, qe in zip(chunk, q):
                        cache[e] = qe
        return [cache[e] for e in locals_]

    def forward_nvfp4(self, tokens, x_gscale: float, h_gscale: float, want_y: bool = False):
        """The oracle's NVFP4 forward of `tokens` (threaded over tokens)."""
        c = self.cfg
        tokens = np.asarray(tokens, np.int32)
        locs = sorted({self.local_of(int(g)) for t in tokens for g in self.ids[t]} - {-1})
        ws = self.expert_weights_nvfp4(locs)
        wmap = np.full(c.E_local + c.num_shared, -1, np.int32)
        for k, e in enumerate(locs):
            wmap[e] = k
        arrs = [np.stack([w[i] for w in ws]) for i in (0, 1, 3, 4)]
        g1 = np.asarray([w[2] for w in ws], np.float32)
        g2 = np.asarray([w[5] for w in ws], np.float32)

        def run(part):
            return oracle.forward_nvfp4(self.x, self.ids, self.w, wmap, arrs[0], arrs[1], g1, arrs[2], arrs[3], g2,
                                        x_gscale=x_gscale, h_gscale=h_gscale, H=c.hidden, I=c.inter,
                                        E_global=c.E_global, E_local=c.E_local, expert_offset=c.expert_offset,
                                        num_shared=c.num_shared, tokens=part, want_act=True, want_xq=True,
                                        activation=c.activation, act_params=c.act_params, want_y=want_y)

        n = host_threads()
        parts = [p for p in np.array_split(tokens, min(n, max(1, tokens.size))) if p.size]
        if len(parts) <= 1:
            return run(tokens)
        with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
            res = list(ex.map(run, parts))
        return {k: np.concatenate([r[k] for r in res]) for k in res[0]}

    def forward(self, tokens, want_y: bool = False):
        """The oracle's forward of `tokens` (rows of the result follow their
        order), split over all host cores by token."""
        c = self.cfg
        tokens = np.asarray(tokens, np.int32)
        locs = sorted({self.local_of(int(g)) for t in tokens for g in self.ids[t]} - {-1})
        ws = self.expert_weights(locs)
        wmap = np.full(c.E_local + c.num_shared, -1, np.int32)
        for k, e in enumerate(locs):
            wmap[e] = k
        if not locs:  # no local expert at all: any placeholder shapes
            z = np.zeros((1, 2 * c.inter, c.hidden // 2), np.uint8)
            arrs = (z, np.zeros((1, 2 * c.inter, c.hidden // 32), np.uint8),
                    np.zeros((1, c.hidden, c.inter // 2), np.uint8), np.zeros((1, c.hidden, c.inter // 32), np.uint8))
        else:
            arrs = tuple(np.stack([w[i] for w in ws]) for i in range(4))

        def run(part):
            return oracle.forward(self.x, self.ids, self.w, wmap, *arrs, H=c.hidden, I=c.inter, E_global=c.E_global,
                                  E_local=c.E_local, expert_offset=c.expert_offset, num_shared=c.num_shared,
                                  tokens=part, want_act=True, want_xq=True, activation=c.activation,
                                  act_params=c.act_params, want_y=want_y)

        n = host_threads()
        parts = [p for p in np.array_split(tokens, min(n, max(1, tokens.size))) if p.size]
        if len(parts) <= 1:
            return run(tokens)
        with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
            res = list(ex.map(run, parts))
        return {k: np.concatenate([r[k] for r in res]) for k in res[0]}


def host_threads() -> int:
    """Threads for the oracle (its C calls release the GIL)."""
    return max(1, os.cpu_count() or 1)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(bits) -> np.ndarray:
    return synth.bf16_bits_to_f64(bits)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def dense_repeat_bound(shape, ws_split, T: int):
    """Per output element, how far two dense-path results may lie apart.  The
    dense path sums a token's fp32 terms w * Y in no fixed order, so two runs'
    fp32 sums each lie within (k' - 1) * 2^-24 * sum_j |w_j Y_j| of the exact
    sum, then each is rounded to bf16 once.  sum_j |w_j Y_j| comes from the
    split path's rows of the same inputs (the same fp32 products; at 128-row
    tiles rounded to bf16, hence the 2^-7 margin).  Returns M; the bound is
    one bf16 step of the larger result plus 2 k' 2^-24 M (1 + 2^-7)."""
    v = moe.moe_get_views(shape, ws_split)
    kp = shape.kp
    cm = v["c_map"][:T * kp].view(T, kp).long()
    y = v["y"].float()
    M = torch.zeros((T, shape.hidden), dtype=torch.float64, device=y.device)
    for j in range(kp):
        rows = cm[:, j]
        ok = rows >= 0
        M[ok] += y[rows[ok]].abs().double()
    return M.cpu().numpy() * 2 * kp * 2.0 ** -24 * (1 + 2.0 ** -7)


def within_dense_repeat(a, b, slack) -> bool:
    """a, b: bf16 outputs as float64 arrays."""
    step = np.exp2(np.floor(np.log2(np.maximum(np.maximum(np.abs(a), np.abs(b)), 1e-30))) - 7)
    return bool(np.all(np.abs(a - b) <= step + slack))


E4M3_VALUES = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def router_matrix_bits(cfg: synth.MoeConfig) -> np.ndarray:
    """The router matrix as bf16 bits [E_global, H]: the seeded fp32 generator
    (sigma = cfg.router_sigma) rounded to bf16 (RNE) and laid out one expert per row."""
    wr = synth.router_host(cfg)  # fp32 [H, Eg]
    t = torch.from_numpy(np.ascontiguousarray(wr.T)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)
