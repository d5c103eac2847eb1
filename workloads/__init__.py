"""Seeded synthetic inputs for the THD layout-conversion workloads.

This module only draws numbers: document lengths, raw token rows and payload
tensors.  It holds none of the conversion's arithmetic (no partition, route,
label or packing logic), so both the CUDA path's tests/benchmark and the CPU
oracle can take their inputs from it.

Workloads (seed = 1234 + index, the seed of the pages' training runs):

0 ``tiny``        cp=2, documents [8, 12, 4] (T=24), hidden bf16 [24, 2, 4],
                  token ids uniform in [0, 1000).
1 ``lognorm128k`` cp=4, T=131072, document lengths log-normal (median 2048,
                  sigma 1.0, clipped to [1, 32768]) rounded up to a multiple
                  of 8, drawn until the next one would overflow; the remainder
                  is the last document.  Hidden bf16 [T, 16, 128] (4 KiB rows).
2 ``longtail128k`` cp=8, T=131072: one 65536-token document, then uniform
                  lengths in [256, 4096] rounded up to a multiple of 16 until
                  the next would overflow; the remainder closes it.  Hidden bf16
                  [T, 32, 128] (8 KiB rows).
3 ``stress16``    cp=16, 4096 documents with lengths uniform in [32, 512]
                  rounded up to a multiple of 32 (T ~ 1.18 M).  Hidden bf16
                  [T, 256] (512 B rows).
4 ``pipeline``    raw int32 tokens [8, 32768], ids uniform in [0, 151643) so
                  that the EOD id 151643 never occurs by chance, EOD placed
                  after geometric(1/2048) gaps; packed with cp=8 (align 16,
                  pad id 0), MTP depth 3, hidden bf16 [T, 5120] (10 KiB rows).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

SEED = 1234
VOCAB = 151936
EOD_ID = 151643


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    cp: int
    hidden: tuple          # per-row hidden shape (bf16 elements)
    mtp_depth: int = 0
    description: str = ""

    @property
    def row_bytes(self) -> int:
        n = 1
        for h in self.hidden:
            n *= h
        return 2 * n

    @property
    def seed(self) -> int:
        return SEED + self.index


WORKLOADS = [
    Workload(0, "tiny", 2, (2, 4), 0,
             "cp=2, docs [8,12,4], hidden bf16 [24,2,4], ids uniform [0,1000)"),
    Workload(1, "lognorm128k", 4, (16, 128), 0,
             "cp=4, T=131072, log-normal doc lengths (median 2K, max 32K) padded to 8, "
             "hidden bf16 [T,16,128], route reused by 48 layers x 2 swaps"),
    Workload(2, "longtail128k", 8, (32, 128), 0,
             "cp=8, T=131072, one 64K doc + uniform 256-4096 docs padded to 16, "
             "hidden bf16 [T,32,128], fwd+bwd swaps per layer"),
    Workload(3, "stress16", 16, (256,), 0,
             "cp=16, 4096 docs uniform 32-512 padded to 32, hidden bf16 [T,256]"),
    Workload(4, "pipeline", 8, (5120,), 3,
             "raw int32 [8,32768], EOD at geometric(1/2048) gaps, cp=8, MTP depth 3, "
             "hidden bf16 [T,5120]"),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def _round_up(n: int, m: int) -> int:
    return -(-n // m) * m


def _fill_to(rng, total, first, draw, mult):
    lens = list(first)
    used = sum(lens)
    while True:
        L = _round_up(int(draw(rng)), mult)
        if used + L > total:
            break
        lens.append(L)
        used += L
    rest = total - used
    if rest > 0:
        lens.append(rest)
    return lens


def doc_lengths(name: str) -> list:
    """Padded document lengths of workloads 0-3 (each a multiple of 2*cp)."""
    w = BY_NAME[name]
    rng = np.random.Generator(np.random.PCG64(w.seed))
    if name == "tiny":
        return [8, 12, 4]
    if name == "lognorm128k":
        def draw(g):
            v = int(round(float(np.exp(g.normal(np.log(2048.0), 1.0)))))
            return min(max(v, 1), 32768)
        return _fill_to(rng, 131072, [], draw, 8)
    if name == "longtail128k":
        return _fill_to(rng, 131072, [65536], lambda g: int(g.integers(256, 4097)), 16)
    if name == "stress16":
        return [_round_up(int(v), 32) for v in rng.integers(32, 513, size=4096)]
    raise KeyError(f"workload {name!r} has no fixed document lengths")


def boundaries(lengths) -> list:
    """cu_seqlens-style running boundaries [0, l0, l0+l1, ...] of a length list."""
    out = [0]
    for L in lengths:
        out.append(out[-1] + int(L))
    return out


def random_lengths(seed: int, n_docs: int, cp: int, max_chunk: int, empty_frac: float = 0.0) -> list:
    """Small random document lengths for parity cases: multiples of 2*cp with
    1..max_chunk rows per chunk; a share ``empty_frac`` of them is empty."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(n_docs):
        if empty_frac > 0 and rng.random() < empty_frac:
            out.append(0)
        else:
            out.append(2 * cp * int(rng.integers(1, max_chunk + 1)))
    return out


def raw_pipeline_tokens(seed: int = SEED + 4, B: int = 8, S: int = 32768,
                        mean_gap: int = 2048) -> np.ndarray:
    """Raw int32 rows [B, S]: ids uniform in [0, EOD_ID), EOD after each
    geometric(1/mean_gap) gap (gap >= 1), counted from the row start."""
    rng = np.random.Generator(np.random.PCG64(seed))
    raw = rng.integers(0, EOD_ID, size=(B, S), dtype=np.int64).astype(np.int32)
    for b in range(B):
        pos = -1
        while True:
            pos += int(rng.geometric(1.0 / mean_gap))
            if pos >= S:
                break
            raw[b, pos] = EOD_ID
    return raw


def token_ids(seed: int, T: int, high: int = 1000) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, high, size=T, dtype=np.int64).astype(np.int32)


def payload_host(seed: int, T: int, hidden: tuple):
    """bf16 [T, *hidden] ~ N(0, 1) from a seeded CPU torch generator."""
    import torch
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randn((T,) + tuple(hidden), generator=g, dtype=torch.float32).to(torch.bfloat16)


def payload_device(seed: int, T: int, hidden: tuple, device):
    """bf16 [T, *hidden] ~ N(0, 1) drawn on the device from a seeded generator
    (for full-size runs, where drawing on the host would dominate)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn((T,) + tuple(hidden), generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)
