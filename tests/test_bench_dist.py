"""The benchmark's multi-rank bookkeeping on CPU (gloo, world size 2): every
rank times its own microbatch, the slowest rank's time and the sum of all
ranks' bytes make the line rank 0 prints."""

import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp
import torch


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, local = bench.setup_dist(None)
    try:
        dev = torch.device("cpu")
        bench.barrier(w, dev)
        slowest = bench.max_over_ranks(10.0 + 5.0 * r, w, dev)
        total = bench.sum_over_ranks(100.0 * (r + 1), w, dev)
        q.put((r, w, slowest, total))
    finally:
        dist.destroy_process_group()


def test_max_and_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 15.0, 300.0), (1, 2, 15.0, 300.0)]
