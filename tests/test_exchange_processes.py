"""CpExchange end to end with one CP rank per process: the device route
build, libthd's per-rank pack and scatter kernels and the exchange's host
tables, in 2 and 4 processes that share the one GPU here.

The processes' kernels never wait on one another: the all-to-all between
them runs on the host (gloo, over copies of the send and receive buffers,
through CpExchange's all_to_all hook), so the processes only meet in the
collective on the CPU.  Every rank's result in both directions must equal
its shard of the oracle's pack -> all-to-all -> scatter, element by element,
and the round trip must return the shard.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _host_all_to_all(out, inp, output_split_sizes=None, input_split_sizes=None, group=None):
    """all_to_all_single over gloo on host copies of device buffers."""
    recv = torch.empty(out.shape, dtype=out.dtype)
    dist.all_to_all_single(recv, inp.cpu(), output_split_sizes=output_split_sizes,
                           input_split_sizes=input_split_sizes, group=group)
    out.copy_(recv)


def _rank_main(rank, world, port, lens, row_bytes, result_q):
    import oracle
    import context_packed_sequence_gb300 as thd
    import workloads as W

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        cu = W.boundaries(lens)
        T, cp = cu[-1], world
        S = T // cp
        # the whole batch, identical on every rank (seeded), zigzag layout
        x = np.random.default_rng(5).integers(0, 256, size=(T, row_bytes), dtype=np.uint8)
        st = thd.new_status()
        fwd, bwd = thd.route_build_pair(torch.tensor(cu, dtype=torch.int32, device="cuda"), T, cp, status=st)
        ex_f = thd.CpExchange.from_route(fwd, rank, all_to_all=_host_all_to_all)
        ex_b = thd.CpExchange.from_route(bwd, rank, all_to_all=_host_all_to_all)
        shard = torch.from_numpy(x[rank * S:(rank + 1) * S].copy()).cuda()
        y = ex_f(shard)
        z = ex_b(y)
        thd.check_status(st)
        _, _, want = oracle.apply_route(x, oracle.build_route(cu, T, cp, oracle.ZIGZAG_TO_CONTIGUOUS))
        ok = np.array_equal(y.cpu().numpy(), want[rank * S:(rank + 1) * S]) and torch.equal(z, shard)
        result_q.put((rank, bool(ok), ex_f.send_identity, ex_f.recv_identity))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,lens,row_bytes", [
    (2, [8, 12, 4, 36], 48),                          # run engine
    (4, [16, 8, 0, 40, 32, 64, 8], 512),              # bulk engine, an empty document
    (4, [8 * k for k in (5, 1, 9, 2, 2, 7, 1, 1, 3)], 6),  # unit engine
])
def test_cp_exchange_in_processes_sharing_the_gpu(world, lens, row_bytes):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, lens, row_bytes, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(world):
        r, ok, send_id, recv_id = q.get(timeout=300)
        results[r] = (ok, send_id, recv_id)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert all(results[r][0] for r in range(world)), results
    # z->c: every rank's send rows are in order, so packing is skipped everywhere
    assert all(results[r][1] for r in range(world))
