"""Fail-fast checks on the GPU: the device status word must carry the same
failure the oracle raises, in the same order of precedence, without any
trap; downstream kernels must then write nothing.  Also: a corrupted route
index is caught by the kernels' own range check, and route build plus swaps
are captured in a CUDA graph, which any host synchronisation would break."""

import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import thd_oracle as O
import context_packed_sequence_gb300 as thd
from context_packed_sequence_gb300 import _lib as L

pytestmark = pytest.mark.gpu
Z2C, C2Z = O.ZIGZAG_TO_CONTIGUOUS, O.CONTIGUOUS_TO_ZIGZAG


def _oracle_kind(fn, *args):
    try:
        fn(*args)
    except O.ThdValueError as e:
        return e.kind
    return "ok"


BAD_CU = [
    ([4, 8], 8, 2),
    ([0, 8, 4, 8], 8, 2),
    ([0, 6, 8], 8, 2),
    ([0, 8], 16, 2),
    ([4, 2, 3], 8, 2),
    ([0, 6, 4, 9], 8, 2),
    ([0, 6, 16], 8, 2),
    ([0, 4, 4, 12, 10, 16], 16, 2),
    ([0, 8, 16, 24, 30, 32], 32, 2),
]


@pytest.mark.parametrize("cu,T,cp", BAD_CU)
@pytest.mark.parametrize("direction", [Z2C, C2Z])
def test_route_status_matches_oracle(cu, T, cp, direction):
    want = _oracle_kind(oracle.build_route, cu, T, cp, direction)
    assert want != "ok"
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    st = thd.new_status()
    r = thd.route_build(cu_t, T, cp, direction, status=st)
    assert L.STATUS_NAMES[thd.status_read(st)] == want
    # the two-direction build reports the same failure
    stp = thd.new_status()
    thd.route_build_pair(cu_t, T, cp, status=stp)
    assert L.STATUS_NAMES[thd.status_read(stp)] == want
    # the partition kernel reports the same failure
    st2 = thd.new_status()
    thd.partition_indices(cu_t, T, cp, -1, status=st2)
    assert L.STATUS_NAMES[thd.status_read(st2)] == want
    # and a swap given the failed status writes nothing
    x = torch.arange(T * 4, dtype=torch.int32, device="cuda").view(T, 4)
    out = torch.full_like(x, -7)
    thd.swap(x, r, out=out, status=st)
    torch.cuda.synchronize()
    assert bool((out == -7).all())
    with pytest.raises(ValueError):
        thd.check_status(st)


def test_host_errors_raise_at_once():
    cu = torch.tensor([0, 8], dtype=torch.int32, device="cuda")
    with pytest.raises(thd.ThdError) as e:
        thd.route_build(cu, 8, 2, 5)
    assert e.value.kind == "bad_direction"
    with pytest.raises(thd.ThdError) as e:
        thd.route_build(cu, 6, 2, Z2C)
    assert e.value.kind == "invalid_arg"


def test_binding_checks_outputs_and_follows_the_route_status():
    """partition_indices refuses an output of the wrong size; a swap given no
    status word uses the route's, so a route whose build failed moves nothing."""
    cu = torch.tensor([0, 8, 16], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        thd.partition_indices(cu, 16, 2, -1, out=torch.empty(15, dtype=torch.int32, device="cuda"))
    with pytest.raises(TypeError):
        thd.partition_indices(cu, 16, 2, 0, out=torch.empty(8, dtype=torch.int64, device="cuda"))
    got = thd.partition_indices(cu, 16, 2, 0, out=torch.empty(8, dtype=torch.int32, device="cuda"))
    assert got.tolist() == oracle.partition_indices([0, 8, 16], 16, 2, 0)

    bad = thd.route_build(torch.tensor([0, 6, 16], dtype=torch.int32, device="cuda"), 16, 2, Z2C)
    x = torch.arange(16 * 8, dtype=torch.int32, device="cuda").view(16, 8)
    out = torch.full_like(x, -7)
    thd.swap(x, bad, out=out)
    assert thd.status_read(bad.status) == L.ERR_LEN_NOT_DIVISIBLE
    assert bool((out == -7).all())
    good = thd.route_build(cu, 16, 2, Z2C)
    assert torch.equal(thd.swap(x, good), x[good.src_of_dst.long()])


def test_pair_refuses_swapped_directions():
    cu = torch.tensor([0, 8], dtype=torch.int32, device="cuda")
    fwd, bwd = thd.Route(8, 2, Z2C), thd.Route(8, 2, C2Z)
    with pytest.raises(thd.ThdError) as e:
        thd.route_build_pair(cu, 8, 2, routes=(bwd, fwd))
    assert e.value.kind == "bad_direction"


def test_ulysses_host_checks():
    lib = L.load()
    x = torch.zeros(8, 64, dtype=torch.uint8, device="cuda")
    y = torch.empty_like(x)
    s = torch.cuda.current_stream().cuda_stream
    assert lib.thd_ulysses_swap(x.data_ptr(), y.data_ptr(), 8, 2, 64, 5, None, s) == L.ERR_BAD_DIRECTION
    assert lib.thd_ulysses_swap(x.data_ptr(), y.data_ptr(), 8, 3, 64, 0, None, s) == L.ERR_INVALID_ARG   # 8 % 3
    assert lib.thd_ulysses_swap(x.data_ptr(), y.data_ptr(), 8, 2, 63, 0, None, s) == L.ERR_INVALID_ARG   # row % cp
    assert lib.thd_ulysses_swap(x.data_ptr(), x.data_ptr() + 64, 8, 2, 64, 0, None, s) == L.ERR_INVALID_ARG


def test_label_status_matches_oracle():
    cases = [
        ([1, 2, 3, 4], [0, 5], [0, 4]),
        ([1, 2, 3, 4], [0, 2], [0, 8]),
        ([1, 2, 3, 4], [1, 2], [0, 4]),
        ([1, 2, 3, 4], [0, 3, 1], [0, 2, 4]),
        ([1, 2, 3, 4], [0, 1, 2], [0, 3, 2]),
    ]
    for tokens, cu_v, cu in cases:
        want = _oracle_kind(oracle.roll_labels, tokens, cu_v, cu, 1)
        st = thd.new_status()
        dev = lambda v: torch.tensor(v, dtype=torch.int32, device="cuda")
        thd.roll_labels(dev(tokens), dev(cu_v), dev(cu), 1, status=st)
        assert L.STATUS_NAMES[thd.status_read(st)] == want, (tokens, cu_v, cu)


def test_zigzag_label_status_matches_oracle():
    cases = [
        ([1, 2, 3, 4, 5, 6, 7, 8], [0, 3, 8], [0, 4, 8], 2),      # fine
        ([1, 2, 3, 4, 5, 6, 7, 8], [0, 3, 8], [0, 2, 8], 2),      # padded length 2 not a multiple of 4
        ([1, 2, 3, 4, 5, 6, 7, 8], [0, 5, 6], [0, 4, 8], 2),      # valid exceeds padded
        ([1, 2, 3, 4, 5, 6, 7, 8], [0, 3, 2], [0, 4, 8], 2),      # unpadded not monotone
    ]
    dev = lambda v: torch.tensor(v, dtype=torch.int32, device="cuda")
    for tokens, cu_v, cu, cp in cases:
        want = _oracle_kind(oracle.roll_labels_zigzag, tokens, cu_v, cu, cp, 0)
        st = thd.new_status()
        thd.roll_labels_zigzag(dev(tokens), dev(cu_v), dev(cu), cp, 0, status=st)
        assert L.STATUS_NAMES[thd.status_read(st)] == want, (cu_v, cu)


def test_status_is_sticky_until_cleared():
    good = torch.tensor([0, 8, 16], dtype=torch.int32, device="cuda")
    bad = torch.tensor([0, 6, 16], dtype=torch.int32, device="cuda")
    st = thd.new_status()
    thd.route_build(bad, 16, 2, Z2C, status=st)
    r = thd.route_build(good, 16, 2, Z2C, status=st)      # skipped: status already set
    assert thd.status_read(st) == L.ERR_LEN_NOT_DIVISIBLE
    thd.status_clear(st)
    r = thd.route_build(good, 16, 2, Z2C, status=st, route=r)
    assert thd.status_read(st) == L.OK
    assert r.src_of_dst.cpu().tolist() == oracle.build_route([0, 8, 16], 16, 2, Z2C).src_of_dst


@pytest.mark.parametrize("cp,heads,head_bytes", [(16, 16, 32), (8, 32, 256)])
def test_ulysses_skips_when_status_is_set(cp, heads, head_bytes):
    """A set status word makes the exchange a no-op (tile transpose and bulk
    row engine alike); after clearing it the exchange runs."""
    x = torch.randint(0, 256, (64, heads, head_bytes), dtype=torch.uint8, device="cuda")
    out = torch.full((cp, 64, heads // cp, head_bytes), 7, dtype=torch.uint8, device="cuda")
    st = thd.new_status()
    thd.route_build(torch.tensor([0, 6, 16], dtype=torch.int32, device="cuda"), 16, 2, Z2C, status=st)
    thd.ulysses_swap(x, cp, thd.SEQ_TO_HEAD, out=out, status=st)
    assert thd.status_read(st) == L.ERR_LEN_NOT_DIVISIBLE
    assert bool((out == 7).all())
    thd.status_clear(st)
    thd.ulysses_swap(x, cp, thd.SEQ_TO_HEAD, out=out, status=st)
    assert thd.status_read(st) == L.OK
    assert torch.equal(thd.ulysses_swap(out, cp, thd.HEAD_TO_SEQ), x)


@pytest.mark.parametrize("tokens_capacity,ok", [(15, False), (16, True), (64, True)])
def test_pack_docs_reports_a_too_small_output(tokens_capacity, ok):
    """Two documents of 4 and 2 tokens padded to multiples of 8 need 16 output
    tokens: with room for 15 the device reports THD_ERR_CAPACITY and writes no
    document; with 16 or more the packing matches the oracle."""
    raw = [[1, 2, 3, 99, 4, 5]]
    kw = dict(tokens_capacity=tokens_capacity)
    if not ok:
        with pytest.raises(thd.ThdError) as e:
            thd.pack_docs(torch.tensor(raw, dtype=torch.int32, device="cuda"), 99, 8, **kw)
        assert e.value.kind == "capacity"
        return
    tok, cu_v, cu = thd.pack_docs(torch.tensor(raw, dtype=torch.int32, device="cuda"), 99, 8, **kw)
    want = oracle.pack_docs(raw, 99, 8)
    assert (tok.cpu().tolist(), cu_v.cpu().tolist(), cu.cpu().tolist()) == tuple(want)


def test_pack_docs_capacity_with_many_chunks():
    """Above 512 chunks the capacity check runs in the separate scan kernel:
    two rows of just over 2^20 tokens (1026 chunks) need T output tokens;
    room for T - 1 raises THD_ERR_CAPACITY, room for exactly T packs."""
    rng = np.random.default_rng(91)
    raw = rng.integers(1, 50, size=(2, 2**20 + 123)).astype(np.int32)
    raw[rng.random(raw.shape) < 1 / 2500] = 99
    T = len(oracle.pack_docs(raw.tolist(), 99, 16)[0])
    x = torch.from_numpy(raw).cuda()
    with pytest.raises(thd.ThdError) as e:
        thd.pack_docs(x, 99, 16, tokens_capacity=T - 1)
    assert e.value.kind == "capacity"
    tok, cu_v, cu = thd.pack_docs(x, 99, 16, tokens_capacity=T)
    assert tok.numel() == T and int(cu[-1]) == T


@pytest.mark.skipif(os.environ.get("THD_CHECKED") != "1", reason="the debug request is in the checked build only")
@pytest.mark.parametrize("width", [1024, 8])
def test_bulk_wait_that_runs_out_reports_timeout(width):
    """Block 0 of a bulk swap waits for 16 bytes that never come: its bounded
    wait gives up (about 3 s), the block lets its other copies land and
    records THD_ERR_TIMEOUT; the next swap on the same context is exact.
    4 KiB rows take the bulk engine, 32 B rows the run engine."""
    lib = L.load()
    stall = lib.thd_debug_stall_next_bulk_copy
    stall.restype, stall.argtypes = ctypes.c_int, [ctypes.c_void_p]
    cu = torch.tensor([0, 8, 20, 24], dtype=torch.int32, device="cuda")
    r = thd.route_build(cu, 24, 2, Z2C)
    x = torch.arange(24 * width, dtype=torch.int32, device="cuda").view(24, width)
    want = x[r.src_of_dst.long()]
    st = thd.new_status()
    assert stall(torch.cuda.current_stream().cuda_stream) == L.OK
    thd.swap(x, r, status=st)
    assert thd.status_read(st) == L.ERR_TIMEOUT
    thd.status_clear(st)
    out = thd.swap(x, r, status=st)
    assert thd.status_read(st) == L.OK
    assert torch.equal(out, want)


@pytest.mark.skipif(os.environ.get("THD_CHECKED") != "1", reason="the debug request is in the checked build only")
@pytest.mark.parametrize("direction", [thd.SEQ_TO_HEAD, thd.HEAD_TO_SEQ])
def test_ulysses_tile_wait_that_runs_out_reports_timeout(direction):
    """Block 0 of the tile transpose waits on its first buffer for 16 bytes
    that never come: sequence -> head gives up as one block, head -> sequence
    through its loading warp and transposing warps; either way the status
    says THD_ERR_TIMEOUT and the next exchange on the same context is exact."""
    lib = L.load()
    stall = lib.thd_debug_stall_next_ulysses_tile
    stall.restype, stall.argtypes = ctypes.c_int, [ctypes.c_void_p]
    cp, T = 16, 4096
    x = torch.randint(0, 256, (T, cp, 32), dtype=torch.uint8, device="cuda")     # 32-byte head groups
    src = x if direction == thd.SEQ_TO_HEAD else thd.ulysses_swap(x, cp, thd.SEQ_TO_HEAD)
    want = thd.ulysses_swap(src, cp, direction)
    st = thd.new_status()
    assert stall(torch.cuda.current_stream().cuda_stream) == L.OK
    thd.ulysses_swap(src, cp, direction, status=st)
    assert thd.status_read(st) == L.ERR_TIMEOUT
    thd.status_clear(st)
    assert torch.equal(thd.ulysses_swap(src, cp, direction, status=st), want)
    assert thd.status_read(st) == L.OK


@pytest.mark.parametrize("width", [8, 128, 4096, 12288])
def test_corrupted_route_index_is_range_checked(width):
    """An out-of-range entry is skipped by the kernel's own check (the access
    never happens) and reported; every other row still moves.  Widths cover
    the unit engine (32 B rows) and the bulk engine (512 B, 16 KiB rows and
    48 KiB rows cut into pieces)."""
    cu = [0, 8, 20, 24]
    r = thd.route_build(torch.tensor(cu, dtype=torch.int32, device="cuda"), 24, 2, Z2C)
    good = r.src_of_dst.clone()
    r.src_of_dst[5] = 24 + 1000
    r.src_of_dst[9] = -3
    x = torch.arange(24 * width, dtype=torch.int32, device="cuda").view(24, width)
    out = torch.full_like(x, -1)
    st = thd.new_status()
    thd.swap(x, r, out=out, status=st)
    assert thd.status_read(st) == L.ERR_INDEX_RANGE
    keep = [q for q in range(24) if q not in (5, 9)]
    assert torch.equal(out[keep], x[good.long()][keep])
    assert bool((out[5] == -1).all()) and bool((out[9] == -1).all())


def test_route_and_swaps_capture_in_a_cuda_graph():
    """Stream capture fails on any synchronising call, so a successful capture
    of route build + swaps shows the path makes no host synchronisation."""
    cu_list = [0, 8, 20, 24, 24, 64]          # lengths 8, 12, 4, 0, 40: multiples of 2*cp
    cu = torch.tensor(cu_list, dtype=torch.int32, device="cuda")
    T, cp = 64, 2
    x = torch.randn(T, 16, device="cuda").to(torch.bfloat16)
    st = thd.new_status()
    fwd = thd.Route(T, cp, Z2C)
    bwd = thd.Route(T, cp, C2Z)
    y = torch.empty_like(x)
    z = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        thd.route_build(cu, T, cp, Z2C, status=st, route=fwd)      # warm-up outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            thd.route_build(cu, T, cp, Z2C, status=st, route=fwd)
            thd.route_build(cu, T, cp, C2Z, status=st, route=bwd)
            thd.swap(x, fwd, out=y, status=st)
            thd.swap(y, bwd, out=z, status=st)
    fwd.src_of_dst.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    assert thd.status_read(st) == L.OK
    assert fwd.src_of_dst.cpu().tolist() == oracle.build_route(cu_list, T, cp, Z2C).src_of_dst
    assert torch.equal(z, x)


def test_full_step_captures_in_a_cuda_graph():
    """Labels in both layouts, the route pair, bulk swaps and the Ulysses tile
    transpose (whose launch sets its shared-memory size and asks for its
    occupancy) captured in one graph and replayed twice.  Packing runs before
    the capture: the caller reads T from it once to size the buffers."""
    E, cp = 99, 2
    raw = torch.tensor([[1, 2, 3, E, 4, 5, E, 0], [6, 7, 8, 9, 10, E, 0, 0]], dtype=torch.int32, device="cuda")
    tok, cu_v, cu = thd.pack_docs(raw, E, 2 * cp)            # T known on the host once, outside capture
    T = tok.numel()
    x = torch.randint(0, 256, (T, 16, 32), dtype=torch.uint8, device="cuda")
    st = thd.new_status()
    fwd, bwd = thd.Route(T, cp, Z2C), thd.Route(T, cp, C2Z)
    out = {}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def step():
        thd.route_build_pair(cu, T, cp, status=st, routes=(fwd, bwd))
        out["labels"] = thd.roll_labels(tok, cu_v, cu, 1, status=st)
        out["zigzag_labels"] = thd.roll_labels_zigzag(tok, cu_v, cu, cp, 1, status=st)
        out["y"] = thd.swap(x, fwd, status=st)
        out["heads"] = thd.ulysses_swap(out["y"], cp, thd.SEQ_TO_HEAD, status=st)
        out["seq"] = thd.ulysses_swap(out["heads"], cp, thd.HEAD_TO_SEQ, status=st)
        out["back"] = thd.swap(out["seq"], bwd, status=st)

    with torch.cuda.stream(s):
        step()                                                 # warm-up outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
    for _ in range(2):
        out["back"].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert thd.status_read(st) == L.OK
        assert torch.equal(out["back"], x)
    cu_l, cu_v_l, tok_l = cu.cpu().tolist(), cu_v.cpu().tolist(), tok.cpu().tolist()
    o = oracle.build_route(cu_l, T, cp, Z2C)
    assert torch.equal(out["y"].cpu(), x.cpu()[torch.tensor(o.src_of_dst)])
    want = oracle.ulysses_swap(out["y"].cpu().numpy().reshape(T, -1), cp, oracle.SEQ_TO_HEAD)
    assert (out["heads"].cpu().numpy().reshape(cp * T, -1) == want).all()
    assert [t.cpu().tolist() for t in out["labels"]] == list(oracle.roll_labels(tok_l, cu_v_l, cu_l, 1))
    assert [t.cpu().tolist() for t in out["zigzag_labels"]] == list(
        oracle.roll_labels_zigzag(tok_l, cu_v_l, cu_l, cp, 1))


def test_python_layer_makes_no_torch_sync():
    cu = torch.tensor([0, 16, 48], dtype=torch.int32, device="cuda")
    x = torch.randn(48, 32, device="cuda")
    torch.cuda.synchronize()
    prev = torch.cuda.get_sync_debug_mode()
    torch.cuda.set_sync_debug_mode("error")
    try:
        st = thd.new_status()
        r = thd.route_build(cu, 48, 4, Z2C, status=st)
        b = thd.route_build(cu, 48, 4, C2Z, status=st)
        y = thd.swap(thd.swap(x, r, status=st), b, status=st)
    finally:
        torch.cuda.set_sync_debug_mode(prev)
    assert torch.equal(y, x)
