"""The oracle's route driven through a real all-to-all collective (gloo, CPU).

Each process is one context-parallel rank holding its own shard.  It packs
with ``send_rows``, exchanges with ``all_to_all_single`` using the route's
split sizes -- the collective the pages call ([PR273] 2.1) -- and scatters with
``recv_rows``.  The result must be exactly the target layout's shard.  This
pins the reading that send buffers are destination-major and receive buffers
source-major, which is what the collective itself does.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from oracle import thd_oracle as O


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, cu, result_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T = cu[-1]
        S = T // world
        zz = O.zigzag_partition(cu, world)
        # payload row of global token g: (g, 1000 + g)
        mine_z = torch.tensor([[g, 1000 + g] for g in zz[rank]], dtype=torch.int64).reshape(S, 2)
        ok = True
        for direction, shard, want in (
                (O.ZIGZAG_TO_CONTIGUOUS, mine_z,
                 [[g, 1000 + g] for g in range(rank * S, (rank + 1) * S)]),
                (O.CONTIGUOUS_TO_ZIGZAG,
                 torch.tensor([[g, 1000 + g] for g in range(rank * S, (rank + 1) * S)],
                              dtype=torch.int64).reshape(S, 2),
                 [[g, 1000 + g] for g in zz[rank]])):
            rt = oracle.build_route(cu, T, world, direction)
            send = shard[torch.tensor(rt.send_rows[rank], dtype=torch.long)] if S else shard
            recv = torch.empty_like(send)
            dist.all_to_all_single(recv, send, rt.output_split_sizes[rank], rt.input_split_sizes[rank])
            out = torch.empty_like(recv)
            if S:
                out[torch.tensor(rt.recv_rows[rank], dtype=torch.long)] = recv
            ok = ok and out.tolist() == want
        result_q.put((rank, ok))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,lens", [(2, [8, 12, 4]), (2, [4, 0, 28]), (4, [16, 8, 0, 40, 32])])
def test_route_through_real_all_to_all(world, lens):
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, cu, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(results[r] for r in range(world)), results
