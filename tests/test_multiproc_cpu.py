"""Multi-process paths on CPU, as two gloo ranks (spawned processes,
rendezvous on 127.0.0.1):
  - the bench's rank discovery, the barrier around the timed region and the
    max-over-ranks reduction of the step time (each rank runs an independent
    replica of the layer);
  - the layer's one exchange under expert parallelism: each rank computes its
    expert slice (expert_offset) with the oracle and one all-reduce of the
    partial outputs gives the full layer."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_info()
        bench.barrier(w)
        # each rank's mean step time; the bench reports the slowest rank's
        worst = bench.allreduce_max(1.25 + rank, w, "cpu")
        bench.barrier(w)
        q.put((r, w, local, worst))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_barrier_and_max_time(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0] * world, codes
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert [g[0] for g in got] == list(range(world))
    assert all(g[1] == world and g[2] == g[0] for g in got)
    assert all(g[3] == 1.25 + world - 1 for g in got)


def _ep_rank_main(rank, world, port, q):
    """Rank r owns experts [r * E / world, (r + 1) * E / world): the layer's
    expert-parallel slice (expert_offset), computed by the oracle; one
    all-reduce sums the partial [T, H] outputs."""
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    import synth

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        E, T, H, I, k = 8, 5, 64, 64, 3
        cfg = synth.MoeConfig("ep", 13, T=T, E_global=E, E_local=E, expert_offset=0, top_k=k, num_shared=0,
                              hidden=H, inter=I, block_n=16)
        x = synth.x_host(cfg)
        ids, w = oracle.route(synth.logits_host(cfg), k)  # every rank routes over all experts
        q1 = [oracle.quantize_mxfp4(a) for a in synth.w1_host(cfg, cfg.global_ids)]
        q2 = [oracle.quantize_mxfp4(a) for a in synth.w2_host(cfg, cfg.global_ids)]
        El = E // world
        mine = range(rank * El, (rank + 1) * El)
        part = oracle.forward(x, ids, w, np.arange(El, dtype=np.int32), np.stack([q1[e][0] for e in mine]),
                              np.stack([q1[e][1] for e in mine]), np.stack([q2[e][0] for e in mine]),
                              np.stack([q2[e][1] for e in mine]), H=H, I=I, E_global=E, E_local=El,
                              expert_offset=rank * El, num_shared=0)["out_f64"]
        t = torch.from_numpy(np.ascontiguousarray(part))
        dist.all_reduce(t)
        full = oracle.forward(x, ids, w, np.arange(E, dtype=np.int32), np.stack([a for a, _ in q1]),
                              np.stack([b for _, b in q1]), np.stack([a for a, _ in q2]),
                              np.stack([b for _, b in q2]), H=H, I=I, E_global=E, E_local=E, expert_offset=0,
                              num_shared=0)["out_f64"]
        err = float(np.max(np.abs(t.numpy() - full)) / max(np.max(np.abs(full)), 1e-30))
        q.put((rank, err, float(np.abs(part).sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_expert_parallel_slices_all_reduce_to_the_full_layer():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ep_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0] * world, codes
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert [g[0] for g in got] == list(range(world))
    assert all(g[1] <= 1e-12 for g in got), got  # fp64 sums in another order only
    assert all(g[2] > 0 for g in got)  # both slices contribute
