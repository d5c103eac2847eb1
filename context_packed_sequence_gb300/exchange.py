"""The layout conversion between GPUs: one context-parallel rank per process.

"[Task32] feat: fla mcore chunkwise cp stage 3" (Relax PR #273), section 2.1:
each CP rank packs its rows into a send buffer grouped by destination rank,
exchanges them with one all-to-all whose input and output split sizes come
from the route, and scatters what it receives into its own shard.
Section 2.2: a rank whose rows are the identity skips the copy (zero-copy).

Every GPU builds the same route, for all ranks, from the same boundaries
(libthd's device route build: no host synchronisation).  A collective needs
its split sizes on the host, so this rank's row of the split tables, its two
identity flags and the route's status word are copied to the host once per
microbatch and route (one synchronisation, the pages' own design).  Pack and
scatter run in libthd's per-rank kernels (thd_pack_rank, thd_scatter_rank);
the exchange is torch.distributed's all_to_all_single, which NCCL runs as one
group of point-to-point sends and receives between the GPUs.
"""

from __future__ import annotations

import torch
import torch.distributed as dist


class CpExchange:
    """One direction of the layout conversion for rank ``cp_rank``.

    Calling it with this rank's shard of the source layout ([S, ...] rows)
    returns its shard of the target layout.  ``pack`` and ``scatter`` map
    (tensor, out or None) -> tensor; from_route binds libthd's per-rank
    kernels to them.  ``all_to_all`` is the collective, called as
    all_to_all(out, inp, output_split_sizes=..., input_split_sizes=...,
    group=...); by default torch.distributed.all_to_all_single."""

    def __init__(self, cp_rank: int, input_split_sizes, output_split_sizes, send_identity: bool,
                 recv_identity: bool, pack, scatter, group=None, all_to_all=None):
        self.cp_rank = int(cp_rank)
        self.input_split_sizes = [int(v) for v in input_split_sizes]
        self.output_split_sizes = [int(v) for v in output_split_sizes]
        if len(self.input_split_sizes) != len(self.output_split_sizes):
            raise ValueError("input and output split sizes differ in length")
        self.rows = sum(self.input_split_sizes)
        if sum(self.output_split_sizes) != self.rows or min(self.input_split_sizes + self.output_split_sizes,
                                                             default=0) < 0:
            raise ValueError("split sizes must be non-negative and send and receive the same number of rows")
        self.send_identity = bool(send_identity)
        self.recv_identity = bool(recv_identity)
        self._pack, self._scatter = pack, scatter
        self.group = group
        self._all_to_all = all_to_all if all_to_all is not None else dist.all_to_all_single

    @classmethod
    def from_route(cls, route, cp_rank: int, group=None, stream=None, all_to_all=None) -> "CpExchange":
        """Read this rank's split sizes and identity flags from a device
        route (one synchronisation of ``stream``) and bind libthd's per-rank
        pack and scatter.  Raises ThdError when the route's build recorded an
        error."""
        from . import api

        r = int(cp_rank)
        if not 0 <= r < route.cp:
            raise ValueError(f"cp_rank must be in [0, {route.cp}), got {cp_rank}")
        s = stream if stream is not None else torch.cuda.current_stream(route.device)
        # the small tables sit after the three row arrays in the route's
        # buffer: one copy from the first split size to the last flag
        base = route._buf.data_ptr()
        lo = route.c.input_split_sizes - base
        hi = route.c.recv_identity + route.cp - base
        tables = torch.empty(hi - lo, dtype=torch.uint8, pin_memory=True)
        status = torch.zeros(1, dtype=torch.int32, pin_memory=True)
        with torch.cuda.stream(s):
            tables.copy_(route._buf[lo:hi], non_blocking=True)
            if getattr(route, "status", None) is not None:
                status.copy_(route.status, non_blocking=True)
        s.synchronize()
        if int(status[0]) != 0:
            raise api.ThdError(int(status[0]), "CpExchange: the route's build failed")

        def at(addr, n, dtype):
            off = addr - base - lo
            size = torch.empty((), dtype=dtype).element_size()
            return tables[off:off + n * size].view(dtype).tolist()

        cp = route.cp
        ins = at(route.c.input_split_sizes + 4 * cp * r, cp, torch.int32)
        outs = at(route.c.output_split_sizes + 4 * cp * r, cp, torch.int32)
        send_id = at(route.c.send_identity + r, 1, torch.uint8)[0]
        recv_id = at(route.c.recv_identity + r, 1, torch.uint8)[0]

        def pack(shard, out):
            return api.pack_rank(shard, route, r, out=out, stream=s)

        def scatter(recv, out):
            return api.scatter_rank(recv, route, r, out=out, stream=s)

        return cls(r, ins, outs, send_id, recv_id, pack, scatter, group, all_to_all)

    def __call__(self, shard: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
        if shard.dim() < 1 or shard.shape[0] != self.rows:
            raise ValueError(f"the shard must have {self.rows} rows, got shape {tuple(shard.shape)}")
        send = shard.contiguous() if self.send_identity else self._pack(shard, None)
        recv = torch.empty_like(send)
        self._all_to_all(recv, send, output_split_sizes=self.output_split_sizes,
                         input_split_sizes=self.input_split_sizes, group=self.group)
        if self.recv_identity:
            if out is None:
                return recv
            out.copy_(recv)
            return out
        return self._scatter(recv, out)
