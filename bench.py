"""Benchmark of the fused MXFP4 MoE layer forward on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

One step = one pass of the whole layer (route -> sort -> x quantise/gather ->
FC1 -> FC2 -> combine) over one batch of synthetic inputs, replayed as one
CUDA graph, inputs resident in HBM, L2 flushed (a 512 MiB memset, then a
256 MiB read of another buffer, outside the timing events) before every step.  Default workload: the decode configuration
(T 32 tokens, 896 experts, top-16, H 3584, I 384, block_n 32, seed 1).

Prints one JSON line (rank 0).  `value` is tokens/s over all ranks (each rank
runs an independent replica of the workload: the layer has no data-parallel
exchange, "replicas only"), `ms_per_step` the mean device time of a step.
`roofline` is for the dominant kernel, timed live with CUDA events on the
launching stream.  `e2e` is the same metric through moe_layer_host with the
inputs copied from pinned host memory and the output copied back inside the
timed region.  `cpu_baseline` times the CPU oracle on a bounded sample.
--impl reference runs the CPU oracle itself (the reference arm).
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
    ap.add_argument("--config", default="decode_t32")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's token count (profiling cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--block-n", type=int, default=0, help="override the workload's virtual-expert rows")
    ap.add_argument("--router", action="store_true",
                    help="start the layer from x and a bf16 router matrix (router GEMM in the chain)")
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


def measured_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu capture of this kernel and
    workload, or None when the GEMM sources changed since the capture."""
    p = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get("%s/%s" % (workload, kernel))
    if not rec or rec.get("gemm_source_hash") != gemm_source_hash():
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
    """nvidia-smi clock/throttle samples while the timed region runs."""

    def __init__(self, index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), "--query-gpu=" + q,
                                       "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            for k, n in enumerate(names):
                if r[5 + k].strip() == "Active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------- ours
def setup_layer(cfg, device):
    import torch

    import mxfp4_mixture_experts_02_gb300 as moe
    import synth

    shape = moe.MoeShape(T=cfg.T, max_T=cfg.T, E_global=cfg.E_global, E_local=cfg.E_local,
                         expert_offset=cfg.expert_offset, top_k=cfg.top_k, num_shared=cfg.num_shared,
                         hidden=cfg.hidden, inter=cfg.inter, block_n=cfg.block_n, shared_scale=cfg.shared_scale,
                         activation=cfg.activation, act_params=tuple(cfg.act_params))
    gids = cfg.global_ids
    E, H, I = gids.size, cfg.hidden, cfg.inter
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


def run_ours(args, cfg):
    import torch

    rank, world, local = dist_info()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    moe, shape, weights, x, logits, sl, ws, ids, tw, out = setup_layer(cfg, device)
    stream = torch.cuda.Stream(device)
    flush = L2Flush(device)

    wr = None
    if args.router:
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
        for _ in range(args.warmup):
            flush()
            g.replay()
        torch.cuda.synchronize()
        st, det = moe.moe_get_status(ws)
        if st != 0:
            raise RuntimeError("device status %d detail %d" % (st, det))

        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        sampler = ClockSampler(local) if rank == 0 else None
        t_wall = time.time()
        for i in range(args.steps):
            flush()
            starts[i].record(stream)
            g.replay()
            ends[i].record(stream)
        torch.cuda.synchronize()
        t_wall = time.time() - t_wall
        barrier(world)
        clocks = sampler.stop() if sampler else None
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = float(np.mean(step_ms))
    ms = allreduce_max(ms, world, device)

    router = time_router(moe, shape, x, wr, ws, logits, flush, stream, max(10, min(args.steps, 200))) if wr is not None \
        else None
    # live per-kernel timing (events between the launches, same stream; in
    # --router mode the logits are the router GEMM's, left by the last step)
    kernel_ms = profile_kernels(moe, shape, weights, x, logits, sl, ws, ids, tw, out, flush, stream,
                                max(10, min(args.steps, 200)))
    # end to end through host buffers
    e2e = run_e2e(moe, shape, weights, cfg, ws, stream, flush, max(10, min(args.steps, 200)))

    hdr = ws[:64 * 4].view(torch.int32).cpu().numpy()
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
    tpeak = 2.0 * bf16
    if flops / (tpeak * 1e12) > dom_bytes / (hbm * 1e9):
        achieved = flops / dt / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                "frac": achieved / tpeak, "traffic": measured_traffic(cfg.name, dom),
                "peak_kind": "%s bf16 burst x 2 (mxf8f6f4, FP8-class)" % peak_kind,
                "frac_of_fp4_peak": achieved / (6.0 * bf16), "algorithmic_flops": flops,
                "algorithmic_bytes": dom_bytes}
    else:
        achieved = dom_bytes / dt / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": measured_traffic(cfg.name, dom), "peak_kind": peak_kind,
                "algorithmic_bytes": dom_bytes, "algorithmic_flops": flops,
                "tensor_frac": flops / dt / 1e12 / tpeak}
    res = {
        "metric": METRIC,
        "value": world * cfg.T / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "us_per_layer": ms * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4 weights x mxfp8 activations, fp32 accumulate, bf16 out",
        "data": "synthetic (seeded Irwin-Hall normal inputs, random-init weights quantised to MXFP4)",
        "config": {"workload": cfg.name, "T": cfg.T, "E_global": cfg.E_global, "E_local": cfg.E_local,
                   "top_k": cfg.top_k, "num_shared": cfg.num_shared, "hidden": H, "inter": I,
                   "block_n": cfg.block_n, "seed": cfg.seed, "activation": ACT_NAMES[cfg.activation],
                   "act_params": list(cfg.act_params), "l2": "flushed before every step (512 MiB memset, then "
                   "a 256 MiB read of another buffer; outside the step events)", "graph": "one CUDA graph per step", "parallelism": "replicas"},
        "layer": {"routed_rows": R, "touched_experts": touched, "weight_bytes_touched": layer_weight_bytes,
                  "hbm_frac_layer": layer_weight_bytes / (ms * 1e-3) / 1e9 / hbm,
                  "tensor_frac_layer": (fc1_flops + fc2_flops) / (ms * 1e-3) / 1e12 / (2.0 * bf16),
                  "kernel_us": {k: kernel_ms[k] * 1e3 for k in names},
                  "fc1": {"bytes": fc1_bytes, "flops": fc1_flops, "gbs": fc1_bytes / kernel_ms["fc1"] / 1e6,
                          "tflops": fc1_flops / kernel_ms["fc1"] / 1e9},
                  "fc2": {"bytes": fc2_bytes, "flops": fc2_flops, "gbs": fc2_bytes / kernel_ms["fc2"] / 1e6,
                          "tflops": fc2_flops / kernel_ms["fc2"] / 1e9}},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": (moe.moe_layer_launch_count(shape) + (1 if wr is not None else 0)) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if router is not None:
        res["router"] = router
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(cfg, budget_s=12.0)
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


def profile_kernels(moe, shape, weights, x, logits, sl, ws, ids, tw, out, flush, stream, reps):
    import torch
    names = ["route", "sort", "gather", "fc1", "fc2", "combine"]
    acc = {k: 0.0 for k in names}
    with torch.cuda.stream(stream):
        for r in range(reps + 3):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
            flush()
            moe.moe_layer_events(shape, logits, sl, x, weights, ws, ids, tw, out, ev)
            torch.cuda.synchronize()
            if r >= 3:
                for k, n in enumerate(names):
                    acc[n] += ev[k].elapsed_time(ev[k + 1])
    return {k: v / reps for k, v in acc.items()}


def run_e2e(moe, shape, weights, cfg, ws, stream, flush, reps):
    import torch

    import synth
    dev = ws.device
    lh = synth.logits_device(cfg, dev).cpu().pin_memory()
    xh = synth.x_device(cfg, dev).cpu().pin_memory()
    sh = synth.shared_logit_device(cfg, dev).contiguous().cpu().pin_memory() if cfg.num_shared else None
    oh = torch.empty((cfg.T, cfg.hidden), dtype=torch.bfloat16).pin_memory()
    times = []
    with torch.cuda.stream(stream):
        for r in range(reps + 3):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            moe.moe_layer_host(shape, lh, sh, xh, weights, ws, oh)
            b.record(stream)
            torch.cuda.synchronize()
            if r >= 3:
                times.append(a.elapsed_time(b))
    ms = float(np.mean(times))
    h2d = lh.numel() * 4 + xh.numel() * 2 + (sh.numel() * 2 if sh is not None else 0)
    return {"value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": oh.numel() * 2}


# --------------------------------------------------------------------- oracle
def oracle_step(cfg, tokens, cache):
    """The oracle on a sample of the workload's tokens: routing of all tokens,
    the sort, then the forward of `tokens` (weights quantised by the oracle,
    cached across steps like resident weights)."""
    import oracle
    import synth
    if "x" not in cache:
        cache["x"] = synth.x_host(cfg)
        cache["logits"] = synth.logits_host(cfg)
        cache["shared"] = synth.shared_logit_host(cfg)
    ids, w = oracle.route(cache["logits"], cfg.top_k, cfg.num_shared, cache["shared"], cfg.shared_scale)
    oracle.sort(ids, cfg.E_global, cfg.E_local, cfg.expert_offset, cfg.num_shared, cfg.block_n)
    loc = set()
    for t in tokens:
        for g in ids[t]:
            if g >= cfg.E_global:
                loc.add(cfg.E_local + int(g) - cfg.E_global)
            elif cfg.expert_offset <= g < cfg.expert_offset + cfg.E_local:
                loc.add(int(g) - cfg.expert_offset)
    loc = sorted(loc)
    wc = cache.setdefault("w", {})
    need = [e for e in loc if e not in wc]
    if need:
        f1 = synth.w1_host(cfg, cfg.global_ids[need])
        f2 = synth.w2_host(cfg, cfg.global_ids[need])
        for k, e in enumerate(need):
            wc[e] = oracle.quantize_mxfp4(f1[k]) + oracle.quantize_mxfp4(f2[k])
    wmap = np.full(cfg.E_local + cfg.num_shared, -1, np.int32)
    for k, e in enumerate(loc):
        wmap[e] = k
    arrs = [np.stack([wc[e][i] for e in loc]) for i in range(4)]
    oracle.forward(cache["x"], ids, w, wmap, *arrs, H=cfg.hidden, I=cfg.inter, E_global=cfg.E_global,
                   E_local=cfg.E_local, expert_offset=cfg.expert_offset, num_shared=cfg.num_shared,
                   tokens=np.asarray(tokens, np.int32), activation=cfg.activation, act_params=cfg.act_params)


def cpu_baseline(cfg, budget_s=12.0):
    """Oracle tokens/s on a bounded sample: whole-batch routing and sort plus
    the forward of a few tokens per step, weights quantised once (resident)."""
    cache = {}
    oracle_step(cfg, [0], cache)  # builds/loads the oracle, caches inputs and one token's experts
    n_tok = 0
    t0 = time.time()
    t = 0
    while time.time() - t0 < budget_s:
        tok = [t % cfg.T]
        oracle_step(cfg, tok, cache)
        n_tok += 1
        t += 1
    dt = time.time() - t0
    return {"value": n_tok / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": "%d single-token steps of %s in %.1f s (routing+sort of all %d tokens each step; "
                      "expert weight quantisation cached)" % (n_tok, cfg.name, dt, cfg.T)}


def run_reference(args, cfg):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    cache = {}
    oracle_step(cfg, [0], cache)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.time()
        oracle_step(cfg, [i % cfg.T], cache)
        if i >= args.warmup:
            times.append(time.time() - t0)
        if i >= args.warmup and sum(times) > 120:
            break
    ms = float(np.mean(times)) * 1e3
    val = 1.0 / (ms * 1e-3)
    res = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world,
           "steps": len(times), "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": cfg.name, "T": cfg.T, "hidden": cfg.hidden, "inter": cfg.inter,
                      "E_global": cfg.E_global, "top_k": cfg.top_k, "block_n": cfg.block_n},
           "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                            "sample": "one token's forward per step (plus routing/sort of the batch)"},
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
    if args.act != "swiglu":
        act = ACT_NAMES.index(args.act)
        cfg = cfg.replace(activation=act, act_params=ACT_DEFAULT_PARAMS[act], name="%s_%s" % (cfg.name, args.act))
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
