"""CpExchange -- the conversion between GPUs, one CP rank per process -- on
CPU ranks over gloo.

Each process is one context-parallel rank holding only its own shard.  The
exchange's bookkeeping is what runs here for real: this rank's input and
output split sizes handed to all_to_all_single, the identity shortcuts
(zero-copy: pack or scatter skipped), shapes and the returned buffer.  The
per-rank pack and scatter, which libthd runs on the GPU, are given as the
definitions send = shard[send_rows[r]] and out[recv_rows[r]] = recv over the
oracle's route (their GPU kernels are compared with the oracle in
test_parity.py).  Every rank's result must equal its shard of the target
layout as the oracle's all-rank pack -> all-to-all -> scatter produces it.
"""

import os
import socket

import numpy as np
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
    from context_packed_sequence_gb300 import CpExchange

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T = cu[-1]
        S = T // world
        # payload row g: (g, 7g, -g) in global order
        x = torch.tensor([[g, 7 * g, -g] for g in range(T)], dtype=torch.int64).reshape(T, 3)
        zz = O.zigzag_partition(cu, world)
        ok, calls = True, []
        for direction in (O.ZIGZAG_TO_CONTIGUOUS, O.CONTIGUOUS_TO_ZIGZAG):
            rt = oracle.build_route(cu, T, world, direction)
            # the source layout's buffer, every rank (as the oracle simulates them)
            src_all = x[torch.tensor([g for r in range(world) for g in zz[r]], dtype=torch.long)] \
                if direction == O.ZIGZAG_TO_CONTIGUOUS else x
            _, _, want_all = oracle.apply_route(src_all.numpy(), rt)
            shard = src_all[rank * S:(rank + 1) * S].clone()

            def pack(t, out, rows=rt.send_rows[rank]):
                calls.append("pack")
                return t[torch.tensor(rows, dtype=torch.long)]

            def scatter(t, out, rows=rt.recv_rows[rank]):
                calls.append("scatter")
                res = torch.empty_like(t) if out is None else out
                res[torch.tensor(rows, dtype=torch.long)] = t
                return res

            ex = CpExchange(rank, rt.input_split_sizes[rank], rt.output_split_sizes[rank], rt.send_identity[rank],
                            rt.recv_identity[rank], pack, scatter)
            got = ex(shard)
            ok = ok and np.array_equal(got.numpy(), want_all[rank * S:(rank + 1) * S])
            # identity ranks take the zero-copy path, the others call the kernels
            ok = ok and (("pack" in calls) != rt.send_identity[rank] or S == 0)
            ok = ok and (("scatter" in calls) != rt.recv_identity[rank] or S == 0)
            calls.clear()
        result_q.put((rank, ok))
    finally:
        dist.destroy_process_group()


def _run(world, cu):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, cu, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(results[r] for r in range(world)), results


def _bounds(lens):
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    return cu


@pytest.mark.parametrize("world,lens", [
    (2, [8, 12, 4]),                     # the hand-derived cp=2 route
    (2, [4, 0, 28]),                     # an empty document
    (4, [16, 8, 0, 40, 32]),
    (4, [8 * k for k in (5, 1, 9, 2, 2, 7, 1, 1, 3)]),
])
def test_cp_exchange_over_gloo(world, lens):
    _run(world, _bounds(lens))


def test_cp_exchange_rejects_inconsistent_splits():
    from context_packed_sequence_gb300 import CpExchange
    with pytest.raises(ValueError):
        CpExchange(0, [3, 1], [2, 1], False, False, None, None)
    with pytest.raises(ValueError):
        CpExchange(0, [3, -1], [1, 1], False, False, None, None)
    ex = CpExchange(0, [2, 2], [1, 3], True, True, None, None)
    with pytest.raises(ValueError):
        ex(torch.zeros(3, 2))
