"""The bench's multi-process path on CPU: two gloo ranks (spawned processes,
rendezvous on 127.0.0.1) exercise the rank discovery, the barrier around the
timed region and the max-over-ranks reduction of the step time that the N-GPU
bench uses (each rank runs an independent replica of the layer)."""
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
