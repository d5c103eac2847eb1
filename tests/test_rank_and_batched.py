"""Per-rank pack / scatter, the exchange's host tables, and the swap along a
sequence dim that is not the first -- GPU against the oracle, element by
element (raw bytes: tolerance 0)."""

import numpy as np
import pytest
import torch

import oracle
from oracle import thd_oracle as O
import context_packed_sequence_gb300 as thd
import workloads as W

pytestmark = pytest.mark.gpu
Z2C, C2Z = O.ZIGZAG_TO_CONTIGUOUS, O.CONTIGUOUS_TO_ZIGZAG


def _cu(lens):
    return W.boundaries(lens)


def _route(cu, T, cp, d):
    st = thd.new_status()
    r = thd.route_build(torch.tensor(cu, dtype=torch.int32, device="cuda"), T, cp, d, status=st)
    thd.check_status(st)
    return r


CASES = [
    # (seed, cp, n_docs, max_chunk, empty_frac)
    (11, 2, 7, 9, 0.0),
    (12, 3, 30, 6, 0.2),
    (13, 4, 60, 12, 0.1),
    (14, 8, 25, 20, 0.0),
    (15, 16, 300, 3, 0.05),
]


@pytest.mark.parametrize("seed,cp,n,mc,empty", CASES)
@pytest.mark.parametrize("row_bytes", [4, 48, 512])
def test_per_rank_pack_scatter_match_the_oracle(seed, cp, n, mc, empty, row_bytes):
    """Every rank packs its own shard, the all-to-all is done on the side by
    the route's split sizes, every rank scatters what it received: the send
    buffers equal the oracle's pack and the result its pack -> all-to-all ->
    scatter, for both directions (unit, run and bulk copy engines)."""
    cu = _cu(W.random_lengths(seed, n, cp, mc, empty))
    T = cu[-1]
    S = T // cp
    rng = np.random.default_rng(seed * 10 + row_bytes)
    x = torch.from_numpy(rng.integers(0, 256, size=(T, row_bytes), dtype=np.uint8)).cuda()
    for d in (Z2C, C2Z):
        o = oracle.build_route(cu, T, cp, d)
        route = _route(cu, T, cp, d)
        st = thd.new_status()
        sends = [thd.pack_rank(x[r * S:(r + 1) * S], route, r, status=st) for r in range(cp)]
        send_o, _, out_o = oracle.apply_route(x.cpu().numpy(), o)
        assert np.array_equal(torch.cat(sends).cpu().numpy(), send_o)
        recvs = [torch.cat([sends[s][o.send_offsets[s][dd]:o.send_offsets[s][dd + 1]] for s in range(cp)])
                 for dd in range(cp)]
        outs = [thd.scatter_rank(recvs[dd], route, dd, status=st) for dd in range(cp)]
        thd.check_status(st)
        assert np.array_equal(torch.cat(outs).cpu().numpy(), out_o), (d, cp, row_bytes)


def test_per_rank_argument_checks():
    cu = _cu([8, 12, 4])
    route = _route(cu, 24, 2, Z2C)
    shard = torch.zeros((12, 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        thd.pack_rank(shard, route, 2)
    with pytest.raises(ValueError):
        thd.scatter_rank(shard[:11], route, 0)
    lib = thd._lib.load()
    import ctypes
    p = shard.data_ptr()
    assert lib.thd_pack_rank(p, p + 8, 0, 16, ctypes.byref(route.c), None, None) == thd._lib.ERR_INVALID_ARG
    assert lib.thd_scatter_rank(p, p + 4096, -1, 16, ctypes.byref(route.c), None, None) == thd._lib.ERR_INVALID_ARG


@pytest.mark.parametrize("cp,lens", [(2, [8, 12, 4]), (4, [16, 8, 0, 40, 32]), (8, [16 * k for k in (9, 1, 3, 4)])])
def test_exchange_tables_from_the_device_route(cp, lens):
    """CpExchange.from_route reads this rank's split sizes and identity flags
    back in one copy: they must be the oracle's, and the bound per-rank
    kernels must pack and scatter like the oracle."""
    cu = _cu(lens)
    T = cu[-1]
    S = T // cp
    x = torch.arange(T * 4, dtype=torch.int32, device="cuda").reshape(T, 4)
    for d in (Z2C, C2Z):
        o = oracle.build_route(cu, T, cp, d)
        route = _route(cu, T, cp, d)
        for r in range(cp):
            ex = thd.CpExchange.from_route(route, r)
            assert ex.input_split_sizes == o.input_split_sizes[r]
            assert ex.output_split_sizes == o.output_split_sizes[r]
            assert ex.send_identity == o.send_identity[r] and ex.recv_identity == o.recv_identity[r]
            got = ex._pack(x[r * S:(r + 1) * S], None)
            want = x[r * S:(r + 1) * S][torch.tensor(o.send_rows[r], dtype=torch.long, device="cuda")]
            assert torch.equal(got, want)


def test_exchange_refuses_a_failed_route():
    cu = torch.tensor([0, 6, 24], dtype=torch.int32, device="cuda")   # 6 is not a multiple of 2*cp = 4
    st = thd.new_status()
    route = thd.route_build(cu, 24, 2, Z2C, status=st)
    with pytest.raises(thd.ThdError) as e:
        thd.CpExchange.from_route(route, 0)
    assert e.value.kind == "len_not_divisible"


SHAPES = [
    # (shape, seq_dim, dtype): rows of 4 B (unit engine), 48 B (run engine), 512 B (bulk engine)
    ((7, None), 1, torch.int32),
    ((5, None, 3, 8), 1, torch.int16),
    ((2, 3, None, 256), 2, torch.bfloat16),
    ((None, 6), 0, torch.int32),
    ((4, None), -1, torch.int32),
]


@pytest.mark.parametrize("shape,seq_dim,dtype", SHAPES)
@pytest.mark.parametrize("cp", [2, 4])
def test_swap_along_seq_dim_matches_the_oracle(shape, seq_dim, dtype, cp):
    """Every block before the sequence dim goes through the same route: for
    each outer index o, out[o] is the oracle's conversion of x[o]."""
    lens = W.random_lengths(21 + cp, 12, cp, 5, 0.1)
    cu = _cu(lens)
    T = cu[-1]
    shp = tuple(T if s is None else s for s in shape)
    g = torch.Generator(device="cpu").manual_seed(cp)
    x = torch.randint(-30000, 30000, shp, generator=g, dtype=torch.int32).to(dtype).cuda()
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    y = thd.zigzag_contiguous_thd_swap(x, cu_d, cp, thd.ZIGZAG_TO_CONTIGUOUS, seq_dim=seq_dim)
    z = thd.zigzag_contiguous_thd_swap(y, cu_d, cp, thd.CONTIGUOUS_TO_ZIGZAG, seq_dim=seq_dim)
    assert y.shape == x.shape and torch.equal(z, x)
    d = seq_dim % x.dim()
    outer = int(np.prod(shp[:d])) if d else 1
    xb = x.cpu().contiguous().view(torch.uint8).reshape(outer, T, -1).numpy()
    yb = y.cpu().contiguous().view(torch.uint8).reshape(outer, T, -1).numpy()
    o = oracle.build_route(cu, T, cp, Z2C)
    for i in range(outer):
        _, _, want = oracle.apply_route(xb[i], o)
        assert np.array_equal(yb[i], want), i


def test_swap_along_seq_dim_launches_only_the_library_kernel():
    """With the route cached, converting a [outer, T, inner] tensor along
    dim 1 launches one libthd kernel and no torch copy kernel."""
    from torch.profiler import ProfilerActivity, profile

    cu = torch.tensor(_cu(W.random_lengths(5, 40, 4, 9, 0.0)), dtype=torch.int32, device="cuda")
    T = int(cu[-1])
    x = torch.randn(3, T, 16, 64, device="cuda").to(torch.bfloat16)
    cache = thd.RouteCache()
    cache.prebuild(cu, T, 4)
    thd.zigzag_contiguous_thd_swap(x, cu, 4, thd.ZIGZAG_TO_CONTIGUOUS, seq_dim=1, cache=cache)
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        y = thd.zigzag_contiguous_thd_swap(x, cu, 4, thd.ZIGZAG_TO_CONTIGUOUS, seq_dim=1, cache=cache)
        torch.cuda.synchronize()
    kernels = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    if not kernels:
        pytest.skip("the profiler recorded no device activity on this machine")
    assert len(kernels) == 1 and "thd::" in kernels[0] and "BatchedSwapMap" in kernels[0], kernels
    o = oracle.build_route(cu.cpu().tolist(), T, 4, Z2C)
    assert torch.equal(y, x[:, torch.tensor(o.src_of_dst, device="cuda").long()])
