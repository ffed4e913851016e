"""Benchmark of the fused MXFP4 MoE layer forward on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME] [--only]

One step = one pass of the whole layer (route -> sort -> x quantise/gather ->
FC1 -> FC2 -> combine) over one batch of synthetic inputs, replayed as one
CUDA graph, inputs resident in HBM, L2 flushed (a 512 MiB memset, then a
256 MiB read of another buffer, outside the timing events) before every step.

The headline workload is the 32768-token prefill (896 experts, top-16, H 3584,
I 384, 128-row tiles, seed 4); ``configs`` in the same JSON line holds the
other four workloads (tiny, decode_t32, ep_slice_t64, skewed_shared_t256),
each with its own step times, per-kernel times, rooflines and end-to-end
figure (``--only`` skips them, ``--config`` picks another headline).

Prints one JSON line (rank 0).  `value` is tokens/s over all ranks (each rank
runs an independent replica of the workload: the layer has no data-parallel
exchange, "replicas only"), `ms_per_step` the mean device time of a step
(median and p10 / p90 beside it).  `roofline` is for the dominant kernel,
timed live with CUDA events on the launching stream; `layer_roofline` is the
whole layer's fraction (touched-expert weight bytes against HBM for the
decode workloads, the layer's MMA flops against the block-scaled tensor peak
for the prefill).  `e2e` is the same metric through moe_layer_host with the
inputs copied from pinned host memory and the output copied back inside the
timed region: for long batches (128-row tiles) consecutive calls streamed on
two caller streams (`single_call` beside it: one call at a time), for the
decode workloads one call at a time.  `cpu_baseline` times the CPU oracle, threaded over tokens on
all host cores, on a bounded sample.  --impl reference runs that oracle
itself (the reference arm).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoE layer tokens/s and µs/layer at 1 GB300; % of HBM (decode) / FP4 tensor (prefill) roofline"
W1_BYTES_PER_EXPERT = lambda H, I: 2 * I * H // 2 + 2 * I * H // 32  # noqa: E731
W2_BYTES_PER_EXPERT = lambda H, I: H * I // 2 + H * I // 32  # noqa: E731


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="prefill_t32768")
    ap.add_argument("--only", action="store_true", help="time the headline workload alone (no configs record)")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's token count (profiling cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--block-n", type=int, default=0, help="override the workload's virtual-expert rows")
    ap.add_argument("--router", action="store_true",
                    help="start the layer from x and a bf16 router matrix (router GEMM in the chain)")
    ap.add_argument("--fmt", default="mxfp8", choices=["mxfp8", "nvfp4"],
                    help="number format: the workloads' MXFP8 x MXFP4, or the NVFP4 variant (128-row tiles)")
    ap.add_argument("--gemm2", default="auto", choices=["auto", "split", "dense"],
                    help="GEMM2 path: the device gate's rule, or one path forced")
    ap.add_argument("--act", default="swiglu", choices=["swiglu", "swiglu_clamp", "situ"],
                    help="FC1 activation: SwiGLU (the workload's), clamped SwiGLU (limit 7) or SiTU (beta 4, lb 25)")
    return ap.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# the GEMM kernel's own sources: a capture's DRAM bytes stand while these are unchanged
GEMM_SOURCES = ["mxfp4_mixture_experts_02_gb300/csrc/gemm.cu", "mxfp4_mixture_experts_02_gb300/csrc/ptx.cuh",
                "mxfp4_mixture_experts_02_gb300/csrc/common.cuh"]


def gemm_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(workload, T, kernel):
    """DRAM bytes per launch from the committed ncu capture of this kernel,
    workload and token count, or None when there is none or the GEMM sources
    changed since the capture."""
    p = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get("%s/%s" % (workload, kernel))
    if not rec or rec.get("T") != T or rec.get("gemm_source_hash") != gemm_source_hash():
        return None
    return rec["dram_bytes_per_launch"]


class L2Flush:
    """Evicts the previous step's data from L2 (129 MB) between steps, outside
    the timed events: a 512 MiB memset, then a 256 MiB read of another buffer,
    so the step starts with an L2 of clean lines that are none of its inputs
    (the memset's dirty lines are written back here, not inside the step)."""

    def __init__(self, device):
        import torch
        self.torch = torch
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=device)
        self.r = torch.ones(64 << 20, dtype=torch.float32, device=device)
        self.acc = torch.zeros((), dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=0, out=self.acc)


class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms from before the first
    warm-up to after the last timed step, each stamped with the host clock;
    summary() keeps the samples that fall inside the timed windows."""

    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        import threading
        self.rows = []
        self.windows = []
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), "--query-gpu=" + q,
                                       "--format=csv,noheader,nounits", "-lms", "50"], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.p.stdout:
            r = [c.strip() for c in line.split(",")]
            if len(r) >= 9:
                self.rows.append((time.time(), r))

    def window(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            self.p.wait()
            self.t.join(timeout=2)

    def summary(self, windows=None):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        wins = self.windows if windows is None else windows
        # a window shorter than the sampling period still gets its nearest sample
        inside = [r for t, r in self.rows if any(a - 0.05 <= t <= b + 0.05 for a, b in wins)]

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in inside if num(r[1]) is not None]
        mx = [num(r[2]) for _, r in self.rows if num(r[2]) is not None]
        reasons = sorted({n for r in inside for k, n in enumerate(self.NAMES) if r[5 + k] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sm), "samples_total": len(self.rows),
                "timed_s": round(sum(b - a for a, b in wins), 3)}


# --------------------------------------------------------------------- ours
# NVFP4 variant: global scales of x (N(0, 1) within +-6: 2688 / 6) and of the
# intermediate (within +-64)
NV_X_GSCALE, NV_H_GSCALE = 448.0, 42.0


def setup_weights_nvfp4(moe, synth, cfg, device):
    """NVFP4 weights of the workload: quantised (per-expert global scales) and packed on the device."""
    import torch
    gids = cfg.global_ids
    E, H, I = gids.size, cfg.hidden, cfg.inter
    c1 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=device)
    c2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=device)
    s1 = torch.empty((E, 2 * I, H // 16), dtype=torch.uint8, device=device)
    s2 = torch.empty((E, H, I // 16), dtype=torch.uint8, device=device)
    g1 = torch.empty(E, dtype=torch.float32, device=device)
    g2 = torch.empty(E, dtype=torch.float32, device=device)
    for c0 in range(0, E, 64):
        ids = gids[c0:c0 + 64]
        n = ids.size
        g1[c0:c0 + n], c1[c0:c0 + n], s1[c0:c0 + n] = moe.moe_quantize_nvfp4(synth.w1_device(cfg, ids, device))
        g2[c0:c0 + n], c2[c0:c0 + n], s2[c0:c0 + n] = moe.moe_quantize_nvfp4(synth.w2_device(cfg, ids, device))
    p1, q1 = moe.moe_pack_weights_nvfp4(c1, s1, True)
    p2, q2 = moe.moe_pack_weights_nvfp4(c2, s2, False)
    del c1, c2, s1, s2
    return moe.MoeWeights(p1, q1, p2, q2), moe.MoeNvfp4(NV_X_GSCALE, NV_H_GSCALE, g1, g2)


def setup_layer(cfg, device, fmt="mxfp8"):
    import torch

    import mxfp4_mixture_experts_02_gb300 as moe
    import synth

    shape = moe.MoeShape(T=cfg.T, max_T=cfg.T, E_global=cfg.E_global, E_local=cfg.E_local,
                         expert_offset=cfg.expert_offset, top_k=cfg.top_k, num_shared=cfg.num_shared,
                         hidden=cfg.hidden, inter=cfg.inter, block_n=cfg.block_n, shared_scale=cfg.shared_scale,
                         activation=cfg.activation, act_params=tuple(cfg.act_params))
    gids = cfg.global_ids
    E, H, I = gids.size, cfg.hidden, cfg.inter
    if fmt == "nvfp4":
        weights, nv = setup_weights_nvfp4(moe, synth, cfg, device)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        x = synth.x_device(cfg, device)
        logits = synth.logits_device(cfg, device)
        sl = synth.shared_logit_device(cfg, device).contiguous() if cfg.num_shared else None
        ws = moe.workspace(shape, device)
        ids = torch.empty((cfg.T, cfg.kp), dtype=torch.int32, device=device)
        tw = torch.empty((cfg.T, cfg.kp), dtype=torch.float32, device=device)
        out = torch.empty((cfg.T, H), dtype=torch.bfloat16, device=device)
        torch.cuda.synchronize()
        return moe, shape, (weights, nv), x, logits, sl, ws, ids, tw, out
    c1 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=device)
    c2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=device)
    s1 = torch.empty((E, 2 * I, H // 32), dtype=torch.uint8, device=device)
    s2 = torch.empty((E, H, I // 32), dtype=torch.uint8, device=device)
    for c0 in range(0, E, 64):
        ids = gids[c0:c0 + 64]
        n = ids.size
        c, s = moe.moe_quantize_mxfp4(synth.w1_device(cfg, ids, device).reshape(n * 2 * I, H))
        c1[c0:c0 + n] = c.reshape(n, 2 * I, H // 2)
        s1[c0:c0 + n] = s.reshape(n, 2 * I, H // 32)
        c, s = moe.moe_quantize_mxfp4(synth.w2_device(cfg, ids, device).reshape(n * H, I))
        c2[c0:c0 + n] = c.reshape(n, H, I // 2)
        s2[c0:c0 + n] = s.reshape(n, H, I // 32)
    p1, q1 = moe.moe_pack_weights(c1, s1, True)
    p2, q2 = moe.moe_pack_weights(c2, s2, False)
    weights = moe.MoeWeights(p1, q1, p2, q2)
    del c1, c2, s1, s2, c, s
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # drop the fp32 generation chunks and row-major copies
    x = synth.x_device(cfg, device)
    logits = synth.logits_device(cfg, device)
    sl = synth.shared_logit_device(cfg, device).contiguous() if cfg.num_shared else None
    ws = moe.workspace(shape, device)
    ids = torch.empty((cfg.T, cfg.kp), dtype=torch.int32, device=device)
    tw = torch.empty((cfg.T, cfg.kp), dtype=torch.float32, device=device)
    out = torch.empty((cfg.T, H), dtype=torch.bfloat16, device=device)
    torch.cuda.synchronize()
    return moe, shape, weights, x, logits, sl, ws, ids, tw, out


def step_stats(step_ms):
    a = np.asarray(step_ms, np.float64)
    return {"ms_mean": float(a.mean()), "ms_median": float(np.median(a)), "ms_p10": float(np.percentile(a, 10)),
            "ms_p90": float(np.percentile(a, 90)), "n": int(a.size)}


def measure_config(args, cfg, device, stream, flush, sampler, steps, warmup, world):
    """One workload: graph-replayed steps (timed), per-kernel events, the
    router GEMM (--router), the host-buffer path; returns the result record."""
    import torch

    nvfp4 = getattr(args, "fmt", "mxfp8") == "nvfp4"
    moe, shape, weights, x, logits, sl, ws, ids, tw, out = setup_layer(cfg, device, "nvfp4" if nvfp4 else "mxfp8")
    moe.moe_set_gemm2_path({"auto": moe.GEMM2_AUTO, "split": moe.GEMM2_SPLIT, "dense": moe.GEMM2_DENSE}[args.gemm2])
    wr = None
    if nvfp4:
        weights, nv = weights

        def layer():
            moe.moe_layer_nvfp4(shape, nv, logits, sl, x, weights, ws, ids, tw, out)
    elif args.router:
        wr = router_matrix(cfg, device)

        def layer():
            moe.moe_layer_router(shape, wr, sl, x, weights, ws, logits, ids, tw, out)
    else:
        def layer():
            moe.moe_layer(shape, logits, sl, x, weights, ws, ids, tw, out)

    with torch.cuda.stream(stream):
        layer()  # also loads the kernels before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            layer()
        for _ in range(warmup):
            flush()
            g.replay()
        torch.cuda.synchronize()
        st, det = moe.moe_get_status(ws)
        if st != 0:
            raise RuntimeError("%s: device status %d detail %d" % (cfg.name, st, det))

        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        barrier(world)
        torch.cuda.synchronize()
        t_wall = time.time()
        for i in range(steps):
            flush()
            starts[i].record(stream)
            g.replay()
            ends[i].record(stream)
        torch.cuda.synchronize()
        t_end = time.time()
        barrier(world)
    if sampler:
        sampler.window(t_wall, t_end)
    stats = step_stats([a.elapsed_time(b) for a, b in zip(starts, ends)])
    ms = allreduce_max(stats["ms_mean"], world, device)
    reps = max(10, min(steps, 200))
    router = time_router(moe, shape, x, wr, ws, logits, flush, stream, reps) if wr is not None else None
    # live per-kernel timing (events between the launches, same stream; in
    # --router mode the logits are the router GEMM's, left by the last step)
    kernel_ms = profile_kernels(moe, shape, weights, x, logits, sl, ws, ids, tw, out, flush, stream, reps,
                                nv if nvfp4 else None)
    e2e = run_e2e(moe, shape, weights, cfg, ws, stream, flush, reps, nv if nvfp4 else None)

    hdr = ws[:64 * 4].view(torch.int32).cpu().numpy()
    moe.moe_set_gemm2_path(moe.GEMM2_AUTO)
    counts = ws_counts(moe, shape, ws)
    touched = int((counts[:cfg.E_local] > 0).sum()) + int(cfg.num_shared > 0 and counts[cfg.E_local:].sum() > 0)
    R = int(hdr[0])
    H, I = cfg.hidden, cfg.inter
    prefill = cfg.block_n == 128
    ybytes = 2 if prefill else 4
    # FC1's x operand: token-order rows gathered per tile (decode tilings: each
    # token's MXFP8 row is read once from HBM, re-reads hit L2), or the
    # expert-ordered rows (128-row tiles: R rows)
    x_rows = cfg.T if not prefill else R
    fc1_bytes = touched * W1_BYTES_PER_EXPERT(H, I) + x_rows * H * 33 // 32 + R * I * 33 // 32
    fc2_bytes = touched * W2_BYTES_PER_EXPERT(H, I) + R * I * 33 // 32 + R * H * ybytes
    fc1_flops = 2.0 * R * H * 2 * I
    fc2_flops = 2.0 * R * I * H
    layer_weight_bytes = touched * (W1_BYTES_PER_EXPERT(H, I) + W2_BYTES_PER_EXPERT(H, I))
    names = ["route", "sort", "gather", "fc1", "fc2", "combine"]
    dom = "fc1" if kernel_ms["fc1"] >= kernel_ms["fc2"] else "fc2"
    hbm, bf16, peak_kind = peaks()
    dt = kernel_ms[dom] * 1e-3
    # A kernel's bound is the larger of its two floors: algorithmic bytes at
    # the measured HBM rate, or algorithmic flops at the block-scaled tensor
    # rate.  kind::mxf8f6f4 (E4M3 x E2M1) runs at the FP8 rate: peak = measured
    # bf16 x 2 (the nominal fp8 : bf16 ratio); the FP4-rate fraction (x 6) is
    # reported beside it.
    dom_bytes = fc1_bytes if dom == "fc1" else fc2_bytes
    flops = fc1_flops if dom == "fc1" else fc2_flops
    # kind::mxf4nvf4 (NVFP4) runs at the FP4 rate: measured bf16 x 6 (nominal 13.5 : 2.25)
    tpeak = (6.0 if nvfp4 else 2.0) * bf16
    if nvfp4:
        # NVFP4 operand bytes: codes half a byte, one scale byte per 16 elements
        wb1 = lambda: 2 * I * H // 2 + 2 * I * H // 16  # noqa: E731
        wb2 = lambda: H * I // 2 + H * I // 16  # noqa: E731
        fc1_bytes = touched * wb1() + x_rows * H * 9 // 16 + R * I * 9 // 16
        fc2_bytes = touched * wb2() + R * I * 9 // 16 + R * H * ybytes
        dom_bytes = fc1_bytes if dom == "fc1" else fc2_bytes
        layer_weight_bytes = touched * (wb1() + wb2())
    if flops / (tpeak * 1e12) > dom_bytes / (hbm * 1e9):
        achieved = flops / dt / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                "frac": achieved / tpeak, "traffic": measured_traffic(cfg.name, cfg.T, dom),
                "peak_kind": ("%s bf16 burst x 6 (mxf4nvf4, FP4-class)" % peak_kind if nvfp4 else
                              "%s bf16 burst x 2 (mxf8f6f4, FP8-class)" % peak_kind),
                "frac_of_fp4_peak": achieved / (6.0 * bf16), "algorithmic_flops": flops,
                "algorithmic_bytes": dom_bytes}
    else:
        achieved = dom_bytes / dt / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": measured_traffic(cfg.name, cfg.T, dom), "peak_kind": peak_kind,
                "algorithmic_bytes": dom_bytes, "algorithmic_flops": flops,
                "tensor_frac": flops / dt / 1e12 / tpeak}
    sec = ms * 1e-3
    if prefill:
        achieved = (fc1_flops + fc2_flops) / sec / 1e12
        layer_roof = {"bound": "tensor", "achieved": achieved, "unit": "TFLOP/s", "peak": tpeak,
                      "frac": achieved / tpeak,
                      "peak_kind": "%s bf16 burst x %d (%s-class)" % (peak_kind, 6 if nvfp4 else 2,
                                                                     "FP4" if nvfp4 else "FP8"),
                      "frac_of_nominal_fp8": achieved / 4500.0, "frac_of_nominal_fp4": achieved / 13500.0,
                      "algorithmic_flops": fc1_flops + fc2_flops}
    else:
        achieved = layer_weight_bytes / sec / 1e9
        layer_roof = {"bound": "hbm", "achieved": achieved, "unit": "GB/s", "peak": hbm, "frac": achieved / hbm,
                      "peak_kind": peak_kind, "frac_of_nominal_8tbs": achieved / 8000.0,
                      "algorithmic_bytes": layer_weight_bytes}
    rec = {
        "workload": cfg.name, "T": cfg.T, "E_global": cfg.E_global, "E_local": cfg.E_local,
        "expert_offset": cfg.expert_offset, "top_k": cfg.top_k, "num_shared": cfg.num_shared, "hidden": H,
        "inter": I, "block_n": cfg.block_n, "seed": cfg.seed, "activation": ACT_NAMES[cfg.activation],
        "gemm2_path": "dense" if hdr[5] == 1 else "split",
        "format": "nvfp4 (E2M1 x E2M1, E4M3 scales per 16, fp32 global scales)" if nvfp4 else
                  "mxfp8 activations x mxfp4 weights (E8M0 scales per 32)",
        "tokens_per_s": world * cfg.T / sec, "us_per_layer": ms * 1e3, "steps": stats,
        "layer": {"routed_rows": R, "touched_experts": touched, "weight_bytes_touched": layer_weight_bytes,
                  "kernel_us": {k: kernel_ms[k] * 1e3 for k in names},
                  "fc1": {"bytes": fc1_bytes, "flops": fc1_flops, "gbs": fc1_bytes / kernel_ms["fc1"] / 1e6,
                          "tflops": fc1_flops / kernel_ms["fc1"] / 1e9},
                  "fc2": {"bytes": fc2_bytes, "flops": fc2_flops, "gbs": fc2_bytes / kernel_ms["fc2"] / 1e6,
                          "tflops": fc2_flops / kernel_ms["fc2"] / 1e9}},
        "roofline": roof, "layer_roofline": layer_roof, "e2e": e2e,
        "gpu_launches": (moe.moe_layer_launch_count(shape) + (1 if wr is not None else 0)) * steps,
    }
    if router is not None:
        rec["router"] = router
    del g, weights, x, logits, sl, ws, ids, tw, out, wr
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_ours(args, cfg):
    import torch

    import synth
    rank, world, local = dist_info()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    stream = torch.cuda.Stream(device)
    flush = L2Flush(device)
    sampler = ClockSampler(local) if rank == 0 else None
    try:
        head = measure_config(args, cfg, device, stream, flush, sampler, args.steps, args.warmup, world)
        head_windows = list(sampler.windows) if sampler else []
        others = {}
        if not args.only:
            for name in synth.CONFIG_ORDER:
                c = synth.CONFIGS[name]
                if name == cfg.name or (args.tokens and name != cfg.name):
                    continue
                if args.fmt == "nvfp4":  # the variant is timed on its headline workload alone
                    continue
                sub_steps = max(args.steps, 50) if c.T <= 256 else args.steps
                n0 = len(sampler.windows) if sampler else 0
                others[name] = measure_config(args, c, device, stream, flush, sampler, sub_steps,
                                              max(args.warmup, 3), world)
                if sampler:
                    others[name]["clocks"] = sampler.summary(sampler.windows[n0:])
    finally:
        if sampler:
            sampler.stop()
    clocks = sampler.summary(head_windows) if sampler else None
    ms = head["us_per_layer"] * 1e-3
    res = {
        "metric": METRIC,
        "value": head["tokens_per_s"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "us_per_layer": head["us_per_layer"],
        "ms_median": head["steps"]["ms_median"],
        "ms_p10": head["steps"]["ms_p10"],
        "ms_p90": head["steps"]["ms_p90"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4 weights x mxfp8 activations, fp32 accumulate, bf16 out",
        "data": "synthetic (seeded Irwin-Hall normal inputs, random-init weights quantised to MXFP4)",
        "config": {k: head[k] for k in ("workload", "T", "E_global", "E_local", "expert_offset", "top_k",
                                        "num_shared", "hidden", "inter", "block_n", "seed", "activation",
                                        "gemm2_path")},
        "layer": head["layer"],
        "roofline": head["roofline"],
        "layer_roofline": head["layer_roofline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": clocks,
    }
    res["config"].update({"l2": "flushed before every step (512 MiB memset, then a 256 MiB read of another "
                                "buffer; outside the step events)", "graph": "one CUDA graph per step",
                          "parallelism": "replicas"})
    if "router" in head:
        res["router"] = head["router"]
    if others:
        res["configs"] = others
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(cfg, budget_s=12.0)
        for name, rec in others.items():  # the smaller workloads: their whole batch
            rec["cpu_baseline"] = cpu_baseline_batch(synth.CONFIGS[name], budget_s=8.0)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


def router_matrix(cfg, device):
    """bf16 router matrix [E_global, H] from the seeded generator, sigma 1/sqrt(H) (logits ~ N(0, 1))."""
    import torch

    import synth
    c = cfg.replace(router_sigma=1.0 / math.sqrt(cfg.hidden))
    return torch.from_numpy(np.ascontiguousarray(synth.router_host(c).T)).to(device).to(torch.bfloat16)


def time_router(moe, shape, x, wr, ws, logits, flush, stream, reps):
    """The router GEMM alone (one graph, L2 flushed before each replay): us, bytes, flops."""
    import torch
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            moe.moe_router(shape, x, wr, ws, logits)
        for _ in range(3):
            flush()
            g.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            flush()
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
    us = float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e3
    T, H, Eg = shape.T, shape.hidden, shape.E_global
    nbytes = Eg * H * 2 + T * H * 2 + T * Eg * 4
    flops = 2.0 * T * H * Eg
    return {"us": us, "bytes": nbytes, "flops": flops, "gbs": nbytes / us / 1e3, "tflops": flops / us / 1e6,
            "note": "includes the status-word reset node before the kernel"}


def ws_counts(moe, shape, ws):
    v = moe.moe_get_views(shape, ws)
    return v["expert_counts"].cpu().numpy()


def profile_kernels(moe, shape, weights, x, logits, sl, ws, ids, tw, out, flush, stream, reps, nv=None):
    import torch
    names = ["route", "sort", "gather", "fc1", "fc2", "combine"]
    acc = {k: 0.0 for k in names}
    with torch.cuda.stream(stream):
        for r in range(reps + 3):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
            flush()
            if nv is not None:
                moe.moe_layer_nvfp4_events(shape, nv, logits, sl, x, weights, ws, ids, tw, out, ev)
            else:
                moe.moe_layer_events(shape, logits, sl, x, weights, ws, ids, tw, out, ev)
            torch.cuda.synchronize()
            if r >= 3:
                for k, n in enumerate(names):
                    acc[n] += ev[k].elapsed_time(ev[k + 1])
    return {k: v / reps for k, v in acc.items()}


def run_e2e(moe, shape, weights, cfg, ws, stream, flush, reps, nv=None):
    import torch

    import synth
    dev = ws.device
    lh = synth.logits_device(cfg, dev).cpu().pin_memory()
    xh = synth.x_device(cfg, dev).cpu().pin_memory()
    sh = synth.shared_logit_device(cfg, dev).contiguous().cpu().pin_memory() if cfg.num_shared else None
    oh = torch.empty((cfg.T, cfg.hidden), dtype=torch.bfloat16).pin_memory()
    if nv is not None:  # the public NVFP4 path: copy in, moe_layer_nvfp4, copy out
        ld, xd = torch.empty_like(lh, device=dev), torch.empty_like(xh, device=dev)
        sd = torch.empty_like(sh, device=dev) if sh is not None else None
        od = torch.empty((cfg.T, cfg.hidden), dtype=torch.bfloat16, device=dev)
        ids = torch.empty((cfg.T, cfg.kp), dtype=torch.int32, device=dev)
        tw = torch.empty((cfg.T, cfg.kp), dtype=torch.float32, device=dev)
    times = []
    with torch.cuda.stream(stream):
        for r in range(reps + 3):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if nv is not None:
                ld.copy_(lh, non_blocking=True)
                xd.copy_(xh, non_blocking=True)
                if sd is not None:
                    sd.copy_(sh, non_blocking=True)
                moe.moe_layer_nvfp4(shape, nv, ld, sd, xd, weights, ws, ids, tw, od)
                oh.copy_(od, non_blocking=True)
            else:
                moe.moe_layer_host(shape, lh, sh, xh, weights, ws, oh)
            b.record(stream)
            torch.cuda.synchronize()
            if r >= 3:
                times.append(a.elapsed_time(b))
    ms = float(np.mean(times))
    h2d = lh.numel() * 4 + xh.numel() * 2 + (sh.numel() * 2 if sh is not None else 0)
    single = {"value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "h2d_bytes_per_step": h2d,
              "d2h_bytes_per_step": oh.numel() * 2, "mode": "one call at a time, L2 flushed before each"}
    if nv is not None or cfg.block_n != 128:
        return single
    streamed = run_e2e_streamed(moe, shape, weights, cfg, ws, lh, sh, xh, oh, max(20, reps))
    streamed.update({"h2d_bytes_per_step": h2d, "d2h_bytes_per_step": oh.numel() * 2, "single_call": single})
    return streamed


def run_e2e_streamed(moe, shape, weights, cfg, ws, lh, sh, xh, oh_ref, steps):
    """Long batches through moe_layer_host back to back, as a server streams
    them: call i on caller stream i % 2 with that stream's own workspace and
    pinned output, no host synchronisation between calls.  Every call copies
    its inputs in and its output out; one call's output copies share the
    full-duplex host link with the next call's input copies while the GPU
    computes.  The timed region spans all the calls (pipeline fill and drain
    included); the inputs (logits + x) are larger than L2, so no flush runs
    between calls.  The outputs are checked bit for bit against the
    one-call-at-a-time output."""
    import torch
    dev = ws.device
    ws2 = moe.workspace(shape, dev)
    wss = [ws, ws2]
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    outs = [torch.empty_like(oh_ref).pin_memory() for _ in range(2)]
    main = torch.cuda.current_stream(dev)

    def issue(n):
        for s in streams:
            s.wait_stream(main)
        for i in range(n):
            with torch.cuda.stream(streams[i % 2]):
                moe.moe_layer_host(shape, lh, sh, xh, weights, wss[i % 2], outs[i % 2])
        for s in streams:
            main.wait_stream(s)

    issue(4)  # warm-up
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    issue(steps)
    b.record(main)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    same = all(torch.equal(o.view(torch.int16), oh_ref.view(torch.int16)) for o in outs)
    del ws2
    torch.cuda.empty_cache()
    return {"value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "mode": "streamed: consecutive calls on two streams, two workspaces", "outputs_match_single_call": same}


# --------------------------------------------------------------------- oracle
class OracleRunner:
    """The CPU oracle on a workload, as it stands: routing and sort of the whole
    batch, then the forward of sampled tokens, one token per thread on all host
    cores (the oracle's C calls release the GIL).  Expert weights are quantised
    by the oracle once, before timing, like resident weights."""

    def __init__(self, cfg):
        import oracle
        import synth
        self.oracle, self.synth, self.cfg = oracle, synth, cfg
        self.threads = max(1, os.cpu_count() or 1)
        self.x = synth.x_host(cfg)
        self.logits = synth.logits_host(cfg)
        self.shared = synth.shared_logit_host(cfg)
        self.wc = {}
        t0 = time.time()
        self.route_sort()
        self.route_sort_s = time.time() - t0

    def route_sort(self):
        c = self.cfg
        self.ids, self.w = self.oracle.route(self.logits, c.top_k, c.num_shared, self.shared, c.shared_scale)
        self.oracle.sort(self.ids, c.E_global, c.E_local, c.expert_offset, c.num_shared, c.block_n)

    def _local(self, g):
        c = self.cfg
        if g >= c.E_global:
            return c.E_local + int(g) - c.E_global
        return int(g) - c.expert_offset if c.expert_offset <= g < c.expert_offset + c.E_local else -1

    def prepare(self, tokens):
        """Quantise (once) the weights of the experts these tokens use."""
        import concurrent.futures
        need = sorted({self._local(g) for t in tokens for g in self.ids[t]} - {-1} - set(self.wc))

        def one(chunk):
            f1 = self.synth.w1_host(self.cfg, self.cfg.global_ids[chunk])
            f2 = self.synth.w2_host(self.cfg, self.cfg.global_ids[chunk])
            return [self.oracle.quantize_mxfp4(f1[k]) + self.oracle.quantize_mxfp4(f2[k]) for k in range(len(chunk))]
        chunks = [need[i:i + 2] for i in range(0, len(need), 2)]
        with concurrent.futures.ThreadPoolExecutor(max_workers=self.threads) as ex:
            for chunk, q in zip(chunks, ex.map(one, chunks)):
                for e, qe in zip(chunk, q):
                    self.wc[e] = qe

    def forward(self, tokens):
        """The forward of `tokens`, one token per thread."""
        import concurrent.futures
        c = self.cfg
        loc = sorted({self._local(g) for t in tokens for g in self.ids[t]} - {-1})
        wmap = np.full(c.E_local + c.num_shared, -1, np.int32)
        for k, e in enumerate(loc):
            wmap[e] = k
        arrs = [np.stack([self.wc[e][i] for e in loc]) for i in range(4)]

        def run(t):
            return self.oracle.forward(self.x, self.ids, self.w, wmap, *arrs, H=c.hidden, I=c.inter,
                                       E_global=c.E_global, E_local=c.E_local, expert_offset=c.expert_offset,
                                       num_shared=c.num_shared, tokens=np.asarray([t], np.int32),
                                       activation=c.activation, act_params=c.act_params)
        with concurrent.futures.ThreadPoolExecutor(max_workers=self.threads) as ex:
            list(ex.map(run, tokens))

    def describe(self, n_tok, fwd_s):
        return ("route + sort of all %d tokens (%.2f s, 1 thread) + the forward of %d tokens, one per thread on %d "
                "threads (%.1f s); tokens/s = 1 / (forward s per token + route/sort s per token); weights quantised "
                "by the oracle beforehand (resident)" % (self.cfg.T, self.route_sort_s, n_tok, self.threads, fwd_s))

    def tokens_per_s(self, n_tok, fwd_s):
        return 1.0 / (fwd_s / n_tok + self.route_sort_s / self.cfg.T)


def cpu_baseline(cfg, budget_s=12.0):
    """Oracle tokens/s on a bounded sample of the workload (see OracleRunner)."""
    r = OracleRunner(cfg)
    n = r.threads
    toks = [t % cfg.T for t in range(4 * n)]
    r.prepare(toks)
    n_tok, fwd_s, i = 0, 0.0, 0
    while fwd_s < budget_s and i < len(toks):
        batch = toks[i:i + n]
        t0 = time.time()
        r.forward(batch)
        fwd_s += time.time() - t0
        n_tok += len(batch)
        i += n
    return {"value": r.tokens_per_s(n_tok, fwd_s), "unit": "tokens/s", "cores": r.threads, "kind": "oracle",
            "sample": r.describe(n_tok, fwd_s)}


def cpu_baseline_batch(cfg, budget_s=8.0):
    """Oracle tokens/s on a whole small batch: its routing and sort, then the
    forward of every token, one token per thread on all host cores (stopping
    early only if the budget runs out, which the sample says)."""
    r = OracleRunner(cfg)
    toks = list(range(cfg.T))
    r.prepare(toks)
    n = r.threads
    n_tok, fwd_s = 0, 0.0
    for i in range(0, len(toks), n):
        if fwd_s >= budget_s:
            break
        batch = toks[i:i + n]
        t0 = time.time()
        r.forward(batch)
        fwd_s += time.time() - t0
        n_tok += len(batch)
    whole = n_tok == cfg.T
    return {"value": r.tokens_per_s(n_tok, fwd_s), "unit": "tokens/s", "cores": r.threads, "kind": "oracle",
            "sample": ("the whole batch: " if whole else "a partial batch: ") + r.describe(n_tok, fwd_s)}


def run_reference(args, cfg):
    """The reference arm: the oracle (the pages hold no runnable code) on the
    host cores, each step a bounded sample of the workload: the forward of one
    token per thread, plus its share of the whole batch's routing and sort."""
    rank, world, _ = dist_info()
    if rank != 0:
        return
    r = OracleRunner(cfg)
    n = r.threads
    total = args.warmup + args.steps
    toks = [t % cfg.T for t in range(total * n)]
    r.prepare(toks)
    times = []
    for i in range(total):
        batch = toks[i * n:(i + 1) * n]
        t0 = time.time()
        r.forward(batch)
        dt = time.time() - t0
        if i >= args.warmup:
            times.append(dt + r.route_sort_s * len(batch) / cfg.T)
        if i >= args.warmup and sum(times) > 150:
            break
    ms = float(np.mean(times)) * 1e3
    val = n / (ms * 1e-3)
    res = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world,
           "steps": len(times), "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": cfg.name, "T": cfg.T, "E_global": cfg.E_global, "E_local": cfg.E_local,
                      "expert_offset": cfg.expert_offset, "top_k": cfg.top_k, "num_shared": cfg.num_shared,
                      "hidden": cfg.hidden, "inter": cfg.inter, "block_n": cfg.block_n, "seed": cfg.seed,
                      "activation": ACT_NAMES[cfg.activation]},
           "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": r.threads, "kind": "oracle",
                            "sample": "per step: " + r.describe(n, float(np.mean(times)))},
           "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(v, world, device):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


ACT_NAMES = ["swiglu", "swiglu_clamp", "situ"]
ACT_DEFAULT_PARAMS = [(0.0, 0.0), (7.0, 0.0), (4.0, 25.0)]


def main():
    args = parse()
    import synth
    cfg = synth.CONFIGS[args.config]
    if args.tokens:
        cfg = cfg.replace(T=args.tokens, name="%s_T%d" % (cfg.name, args.tokens))
    if args.block_n:
        cfg = cfg.replace(block_n=args.block_n, name="%s_B%d" % (cfg.name, args.block_n))
    if args.router:
        cfg = cfg.replace(name="%s_router" % cfg.name)
    if args.fmt == "nvfp4":
        cfg = cfg.replace(name="%s_nvfp4" % cfg.name)
    if args.act != "swiglu":
        act = ACT_NAMES.index(args.act)
        cfg = cfg.replace(activation=act, act_params=ACT_DEFAULT_PARAMS[act], name="%s_%s" % (cfg.name, args.act))
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
