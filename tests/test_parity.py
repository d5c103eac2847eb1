"""GPU vs oracle, element by element (integers and raw bytes: tolerance 0).

Every case is compared in full: small and medium ones against the oracle's
outputs, the full-size workloads' routes entry by entry and their payloads
row by row against the oracle's permutation (plus the round trip z->c->z)."""

import numpy as np
import pytest
import torch

import oracle
from oracle import thd_oracle as O
import context_packed_sequence_gb300 as thd
import workloads as W

pytestmark = pytest.mark.gpu
Z2C, C2Z = O.ZIGZAG_TO_CONTIGUOUS, O.CONTIGUOUS_TO_ZIGZAG


def _cu_tensor(cu):
    return torch.tensor(cu, dtype=torch.int32, device="cuda")


def _gpu_route(cu, T, cp, direction):
    st = thd.new_status()
    r = thd.route_build(_cu_tensor(cu), T, cp, direction, status=st)
    thd.check_status(st, "route_build")
    return r


def _gpu_pair(cu, T, cp, shared=True):
    """Both directions in one launch, into one buffer whose common arrays the
    routes share (Route.pair) or into two separately bound routes."""
    st = thd.new_status()
    routes = None if shared else (thd.Route(T, cp, Z2C), thd.Route(T, cp, C2Z))
    f, b = thd.route_build_pair(_cu_tensor(cu), T, cp, status=st, routes=routes)
    thd.check_status(st, "route_build_pair")
    return f, b


def _assert_both(cu, T, cp):
    """Each direction alone, and both in one launch into a shared and into
    separate buffers, against the oracle; each direction alone into a
    pair-bound buffer leaves the other direction's route intact."""
    want = [oracle.build_route(cu, T, cp, d) for d in (Z2C, C2Z)]
    for d in (Z2C, C2Z):
        _assert_route(_gpu_route(cu, T, cp, d), want[d])
    for shared in (True, False):
        f, b = _gpu_pair(cu, T, cp, shared)
        _assert_route(f, want[Z2C])
        _assert_route(b, want[C2Z])
    st = thd.new_status()
    pf, pb = thd.Route.pair(T, cp)
    thd.route_build(_cu_tensor(cu), T, cp, Z2C, status=st, route=pf)
    thd.route_build(_cu_tensor(cu), T, cp, C2Z, status=st, route=pb)
    thd.check_status(st)
    _assert_route(pf, want[Z2C])
    _assert_route(pb, want[C2Z])
    return want


def _flat(list_of_lists):
    out = []
    for x in list_of_lists:
        out.extend(x)
    return out


def _assert_route(r, o):
    assert r.src_of_dst.cpu().tolist() == o.src_of_dst
    assert r.send_rows.cpu().reshape(-1).tolist() == _flat(o.send_rows)
    assert r.recv_rows.cpu().reshape(-1).tolist() == _flat(o.recv_rows)
    assert r.input_split_sizes.cpu().tolist() == o.input_split_sizes
    assert r.output_split_sizes.cpu().tolist() == o.output_split_sizes
    assert r.send_offsets.cpu().tolist() == o.send_offsets
    assert r.recv_offsets.cpu().tolist() == o.recv_offsets
    assert [bool(v) for v in r.send_identity.cpu().tolist()] == o.send_identity
    assert [bool(v) for v in r.recv_identity.cpu().tolist()] == o.recv_identity


def _bounds(lengths):
    return W.boundaries(lengths)


# --------------------------------------------------------------------------
# route and partition
# --------------------------------------------------------------------------

def test_tiny_workload_route_and_partition():
    lens = W.doc_lengths("tiny")
    cu, cp = _bounds(lens), 2
    T = cu[-1]
    for d in (Z2C, C2Z):
        _assert_route(_gpu_route(cu, T, cp, d), oracle.build_route(cu, T, cp, d))
    st = thd.new_status()
    allr = thd.partition_indices(_cu_tensor(cu), T, cp, -1, status=st)
    one = [thd.partition_indices(_cu_tensor(cu), T, cp, r, status=st) for r in range(cp)]
    thd.check_status(st)
    assert allr.cpu().reshape(-1).tolist() == oracle.partition_indices(cu, T, cp, -1)
    for r in range(cp):
        assert one[r].cpu().tolist() == oracle.partition_indices(cu, T, cp, r)


def _small_packings():
    import itertools
    for cp in (1, 2, 3, 4):
        unit, max_units = 2 * cp, 24 // (2 * cp)
        yield cp, []
        for n in range(1, 4):
            for parts in itertools.product(range(max_units + 1), repeat=n):
                if sum(parts) <= max_units:
                    yield cp, [unit * p for p in parts]


def test_route_bruteforce_small_packings():
    n = 0
    for cp, lens in _small_packings():
        cu = _bounds(lens)
        _assert_both(cu, cu[-1], cp)
        n += 1
    assert n > 250


MEDIUM = [
    # (seed, cp, n_docs, max_chunk, empty_frac)
    (1, 2, 40, 64, 0.1),
    (2, 3, 120, 20, 0.2),
    (3, 4, 300, 12, 0.0),
    (4, 5, 17, 300, 0.3),
    (5, 8, 200, 9, 0.1),
    (6, 16, 150, 5, 0.05),
    (7, 64, 30, 3, 0.0),
    (8, 7, 1, 2000, 0.0),          # one long document
]


@pytest.mark.parametrize("seed,cp,n_docs,max_chunk,empty", MEDIUM)
def test_route_medium(seed, cp, n_docs, max_chunk, empty):
    lens = W.random_lengths(seed, n_docs, cp, max_chunk, empty)
    cu = _bounds(lens)
    T = cu[-1]
    _assert_both(cu, T, cp)
    st = thd.new_status()
    got = thd.partition_indices(_cu_tensor(cu), T, cp, -1, status=st)
    thd.check_status(st)
    assert got.cpu().reshape(-1).tolist() == oracle.partition_indices(cu, T, cp, -1)


@pytest.mark.parametrize("cp,n_docs", [(2, 13000), (64, 4000)])
def test_route_boundaries_beyond_shared_memory(cp, n_docs):
    """Enough documents that the boundaries are searched in global memory."""
    lens = W.random_lengths(99 + cp, n_docs, cp, 2, 0.1)
    cu = _bounds(lens)
    _assert_both(cu, cu[-1], cp)


def test_empty_packing_and_cp1():
    for cu in ([0], [0, 0, 0]):
        _assert_both(cu, 0, 4)
    cu = _bounds([2, 6, 0, 10])
    _assert_both(cu, 18, 1)
    for d in (Z2C, C2Z):
        assert _gpu_route(cu, 18, 1, d).src_of_dst.cpu().tolist() == list(range(18))


# --------------------------------------------------------------------------
# payload movement: fused swap and the three steps, every copy-unit width
# --------------------------------------------------------------------------

def _payload(seed, T, row_bytes):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=(T, row_bytes), dtype=np.uint8)


@pytest.mark.parametrize("row_bytes", [1, 2, 6, 12, 16, 48, 512, 4096])
@pytest.mark.parametrize("seed,cp,n_docs,max_chunk,empty", [MEDIUM[1], MEDIUM[4], (11, 4, 9, 7, 0.2)])
def test_apply_parity(row_bytes, seed, cp, n_docs, max_chunk, empty):
    lens = W.random_lengths(seed, n_docs, cp, max_chunk, empty)
    cu = _bounds(lens)
    T = cu[-1]
    if T * row_bytes > 64 << 20:
        pytest.skip("kept small for the CPU oracle")
    x_np = _payload(seed * 31 + row_bytes, T, row_bytes)
    x = torch.from_numpy(x_np).cuda()
    for d in (Z2C, C2Z):
        o = oracle.build_route(cu, T, cp, d)
        send_o, recv_o, out_o = oracle.apply_route(x_np, o)
        r = _gpu_route(cu, T, cp, d)
        st = thd.new_status()
        out = thd.swap(x, r, status=st)
        send = thd.pack(x, r, status=st)
        recv = thd.a2a_local(send, r, status=st)
        out3 = thd.scatter(recv, r, status=st)
        thd.check_status(st)
        assert np.array_equal(out.cpu().numpy(), out_o)
        assert np.array_equal(send.cpu().numpy(), send_o)
        assert np.array_equal(recv.cpu().numpy(), recv_o)
        assert np.array_equal(out3.cpu().numpy(), out_o)


@pytest.mark.parametrize("row_bytes", [16, 32, 48, 64, 96, 128, 144, 160, 192, 208, 256, 8192, 10240, 20480, 40960])
def test_apply_parity_wide_rows(row_bytes):
    """Every chunk shape of the run engine (16-192 B rows: 16, 8, 4, 2 and 1
    rows per lane, 2 or 3 stages) and every plan of the bulk engine (32 rows
    per chunk, one row per chunk with 2/4/3 stages, rows cut into 16 KiB
    pieces)."""
    for seed, cp, n_docs, max_chunk, empty in [(21, 2, 30, 6, 0.1), (22, 4, 9, 5, 0.2)]:
        lens = W.random_lengths(seed, n_docs, cp, max_chunk, empty)
        cu = _bounds(lens)
        T = cu[-1]
        x_np = _payload(seed * 7 + row_bytes, T, row_bytes)
        x = torch.from_numpy(x_np).cuda()
        for d in (Z2C, C2Z):
            o = oracle.build_route(cu, T, cp, d)
            send_o, recv_o, out_o = oracle.apply_route(x_np, o)
            r = _gpu_route(cu, T, cp, d)
            st = thd.new_status()
            out = thd.swap(x, r, status=st)
            send = thd.pack(x, r, status=st)
            recv = thd.a2a_local(send, r, status=st)
            out3 = thd.scatter(recv, r, status=st)
            thd.check_status(st)
            assert np.array_equal(out.cpu().numpy(), out_o)
            assert np.array_equal(send.cpu().numpy(), send_o)
            assert np.array_equal(recv.cpu().numpy(), recv_o)
            assert np.array_equal(out3.cpu().numpy(), out_o)


def test_unaligned_buffers_take_the_narrow_path():
    """16-byte-multiple rows at a 4-byte offset: correct through the 4-byte units."""
    cu = _bounds(W.random_lengths(31, 25, 2, 9, 0.1))
    T, rb = cu[-1], 512
    x_np = _payload(5, T, rb)
    base = torch.zeros(T * rb + 4, dtype=torch.uint8, device="cuda")
    x = base[4:].view(T, rb)
    x.copy_(torch.from_numpy(x_np))
    obase = torch.zeros(T * rb + 4, dtype=torch.uint8, device="cuda")
    out = obase[4:].view(T, rb)
    for d in (Z2C, C2Z):
        o = oracle.build_route(cu, T, 2, d)
        thd.swap(x, _gpu_route(cu, T, 2, d), out=out)
        assert np.array_equal(out.cpu().numpy(), x_np[o.src_of_dst])


@pytest.mark.parametrize("cp,T,heads,head_bytes", [
    (2, 64, 8, 64),          # 256-byte pieces: tile transpose, one partial tile
    (4, 96, 8, 64),          # 128-byte pieces: tile transpose
    (8, 64, 32, 256),        # 1 KiB pieces, as the 128K workloads: bulk row engine
    (2, 30, 2, 6),           # 6-byte pieces: byte units
    (1, 16, 4, 32),          # cp = 1: a plain copy
    (16, 19984, 16, 32),     # 32-byte pieces: several tiles per block, ragged last tile
    (3, 1503, 3, 48),        # cp = 3, pieces of three 16-byte units, ragged
    (2, 10, 2, 16),          # 16-byte pieces, one partial tile
    (32, 64, 32, 1008),      # rows of 31.5 KiB: one token per tile
    (64, 64, 64, 1008),      # a tile would not fit in shared memory: bulk row engine
    (64, 128, 64, 16),       # cp = 64: each issuing lane takes two runs
    (24, 24 * 411, 24, 32),  # cp = 24: 32/28 KiB tiles, ragged last tile
    (32, 32 * 397, 32, 16),  # cp = 32: 40/32 KiB tiles, ragged last tile
    (64, 64 * 101, 64, 32),  # cp = 64: the 44 KiB tile shrunk to 40 KiB to fit
])
def test_ulysses_parity(cp, T, heads, head_bytes):
    rng = np.random.default_rng(cp * 100 + T)
    x_np = rng.integers(0, 256, size=(T, heads * head_bytes), dtype=np.uint8)
    want = oracle.ulysses_swap(x_np, cp, oracle.SEQ_TO_HEAD)
    x = torch.from_numpy(x_np).cuda().view(T, heads, head_bytes)
    st = thd.new_status()
    y = thd.ulysses_swap(x, cp, thd.SEQ_TO_HEAD, status=st)
    back = thd.ulysses_swap(y, cp, thd.HEAD_TO_SEQ, status=st)
    thd.check_status(st)
    assert tuple(y.shape) == (cp, T, heads // cp, head_bytes)
    assert np.array_equal(y.cpu().numpy().reshape(cp * T, -1), want)
    assert np.array_equal(back.cpu().numpy().reshape(T, -1), oracle.ulysses_swap(want, cp, oracle.HEAD_TO_SEQ))
    assert torch.equal(back, x)


def test_ulysses_fuzz():
    """40 random shapes through every engine of the exchange: cp 1-16, pieces
    of 1-1040 bytes (multiples of 16 below 1 KiB mostly take the tile
    transpose, larger or odd ones the row engines), token counts that leave
    ragged last tiles; both directions against the oracle."""
    rng = np.random.default_rng(2027)
    engines = set()
    for case in range(40):
        cp = int(rng.integers(1, 17))
        if case % 2:
            piece = 16 * int(rng.integers(1, 66))         # 16 .. 1040, mostly the tile transpose
        else:
            piece = int(rng.integers(1, 300))             # any size: run engine (multiples of 16) or unit engine
        T = cp * int(rng.integers(1, max(2, 200000 // (cp * cp * piece + 1))))
        engines.add("tile" if cp > 1 and piece % 16 == 0 and piece < 1024 else "rows")
        x_np = rng.integers(0, 256, size=(T, cp * piece), dtype=np.uint8)
        want = oracle.ulysses_swap(x_np, cp, oracle.SEQ_TO_HEAD)
        x = torch.from_numpy(x_np).cuda().view(T, cp, piece)
        st = thd.new_status()
        y = thd.ulysses_swap(x, cp, thd.SEQ_TO_HEAD, status=st)
        back = thd.ulysses_swap(y, cp, thd.HEAD_TO_SEQ, status=st)
        thd.check_status(st)
        assert np.array_equal(y.cpu().numpy().reshape(cp * T, piece), want), (cp, T, piece)
        assert torch.equal(back, x), (cp, T, piece)
    assert engines == {"tile", "rows"}


@pytest.mark.parametrize("cp,T,piece", [(16, 19984, 32), (3, 1503, 48), (8, 424, 512)])
def test_ulysses_guard_bytes_untouched(cp, T, piece):
    """The tile transpose writes exactly its output: 256 guard bytes on each
    side of the destination keep their pattern in both directions."""
    lib = thd._lib.load()
    row = cp * piece
    x = torch.randint(0, 256, (T, row), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = thd.new_status()
    heads = torch.full((T * row + 512,), 0x5A, dtype=torch.uint8, device="cuda")
    seq = torch.full((T * row + 512,), 0x5A, dtype=torch.uint8, device="cuda")
    assert lib.thd_ulysses_swap(x.data_ptr(), heads.data_ptr() + 256, T, cp, row, thd.SEQ_TO_HEAD,
                                st.data_ptr(), s) == 0
    assert lib.thd_ulysses_swap(heads.data_ptr() + 256, seq.data_ptr() + 256, T, cp, row, thd.HEAD_TO_SEQ,
                                st.data_ptr(), s) == 0
    thd.check_status(st)
    for buf in (heads, seq):
        assert bool((buf[:256] == 0x5A).all()) and bool((buf[256 + T * row:] == 0x5A).all())
    want = oracle.ulysses_swap(x.cpu().numpy(), cp, oracle.SEQ_TO_HEAD)
    assert np.array_equal(heads[256:256 + T * row].cpu().numpy().reshape(cp * T, piece), want)
    assert torch.equal(seq[256:256 + T * row].view(T, row), x)


def test_zigzag_to_ulysses_and_back():
    """Zigzag shards -> contiguous (= Ulysses sequence shards) -> head shards,
    then all the way back, on bf16 hidden states [T, 16, 128]."""
    cu = _bounds(W.random_lengths(77, 30, 4, 20, 0.1))
    T = cu[-1]
    x = W.payload_host(5, T, (16, 128)).cuda()
    fwd, bwd = _gpu_pair(cu, T, 4)
    heads = thd.ulysses_swap(thd.swap(x, fwd), 4, thd.SEQ_TO_HEAD)
    seq = thd.ulysses_swap(heads, 4, thd.HEAD_TO_SEQ)
    assert torch.equal(thd.swap(seq, bwd), x)
    o = oracle.build_route(cu, T, 4, Z2C)
    xc = x.cpu()[torch.tensor(o.src_of_dst)]
    for r in range(4):
        assert torch.equal(heads[r].cpu(), xc[:, 4 * r:4 * (r + 1)])


def test_tiny_workload_payloads():
    """x bf16 [24, 2, 4] and int32 ids, z->c and back, bit for bit."""
    w = W.BY_NAME["tiny"]
    cu = _bounds(W.doc_lengths("tiny"))
    T = cu[-1]
    x = W.payload_host(w.seed, T, w.hidden)
    ids = torch.from_numpy(W.token_ids(w.seed, T)).view(T, 1)
    for t in (x, ids):
        raw = t.contiguous().view(torch.uint8).reshape(T, -1).numpy()
        fwd = oracle.build_route(cu, T, 2, Z2C)
        _, _, want = oracle.apply_route(raw, fwd)
        r = _gpu_route(cu, T, 2, Z2C)
        b = _gpu_route(cu, T, 2, C2Z)
        got = thd.swap(t.cuda(), r)
        back = thd.swap(got, b)
        assert np.array_equal(got.cpu().contiguous().view(torch.uint8).reshape(T, -1).numpy(), want)
        assert torch.equal(back.cpu(), t)


def test_guard_rows_untouched():
    cu = _bounds(W.random_lengths(5, 50, 4, 9, 0.1))
    T = cu[-1]
    r = _gpu_route(cu, T, 4, Z2C)
    x = torch.randint(0, 255, (T, 64), dtype=torch.uint8, device="cuda")
    big = torch.full((T + 64, 64), 0xA5, dtype=torch.uint8, device="cuda")
    out = big[32:32 + T]
    thd.swap(x, r, out=out)
    torch.cuda.synchronize()
    assert bool((big[:32] == 0xA5).all()) and bool((big[32 + T:] == 0xA5).all())
    assert torch.equal(out, x[r.src_of_dst.long()])


def test_guard_bytes_around_route_and_labels_untouched():
    """Route arrays bound inside a larger poisoned buffer, and label outputs
    inside poisoned buffers: nothing outside them is written."""
    import ctypes
    from context_packed_sequence_gb300 import _lib as L
    lib = L.load()
    stream = torch.cuda.current_stream().cuda_stream
    cu = _bounds(W.random_lengths(8, 60, 4, 11, 0.1))
    T, cp, guard = cu[-1], 4, 4096
    cu_d = _cu_tensor(cu)
    nbytes = lib.thd_route_bytes(T, cp)
    blob = torch.full((nbytes + 2 * guard,), 0x5A, dtype=torch.uint8, device="cuda")
    for d in (Z2C, C2Z):
        c = L.ThdRoute()
        assert lib.thd_route_bind(ctypes.byref(c), blob.data_ptr() + guard, nbytes, T, cp, d) == L.OK
        st = thd.new_status()
        assert lib.thd_route_build(cu_d.data_ptr(), len(cu) - 1, T, cp, d, ctypes.byref(c), st.data_ptr(),
                                   stream) == L.OK
        thd.check_status(st)
        assert bool((blob[:guard] == 0x5A).all()) and bool((blob[guard + nbytes:] == 0x5A).all())

    cu_v = _cu_tensor(_bounds([max(0, cu[i + 1] - cu[i] - 3) for i in range(len(cu) - 1)]))
    tokens = torch.arange(T, dtype=torch.int32, device="cuda")
    depth, pad = 2, 32
    for fn, extra in ((lib.thd_roll_labels, ()), (lib.thd_roll_labels_zigzag, (cp,))):
        lab = torch.full(((depth + 1) * T + 2 * pad,), -11, dtype=torch.int32, device="cuda")
        msk = torch.full(((depth + 1) * T + 2 * pad,), 0xEE, dtype=torch.uint8, device="cuda")
        val = torch.full((T + 2 * pad,), 0xEE, dtype=torch.uint8, device="cuda")
        st = thd.new_status()
        assert fn(tokens.data_ptr(), cu_v.data_ptr(), cu_d.data_ptr(), len(cu) - 1, T, *extra, depth, -1, None,
                  None, lab.data_ptr() + 4 * pad, msk.data_ptr() + pad, val.data_ptr() + pad, st.data_ptr(),
                  stream) == L.OK
        thd.check_status(st)
        n = (depth + 1) * T
        assert bool((lab[:pad] == -11).all()) and bool((lab[pad + n:] == -11).all())
        assert bool((msk[:pad] == 0xEE).all()) and bool((msk[pad + n:] == 0xEE).all())
        assert bool((val[:pad] == 0xEE).all()) and bool((val[pad + T:] == 0xEE).all())


def test_route_fuzz_many_cp():
    """Random packings (empty documents included) for cp up to 64, both
    directions in one launch, against the oracle."""
    rng = np.random.default_rng(2024)
    for trial in range(40):
        cp = int(rng.choice([1, 2, 3, 5, 6, 7, 12, 16, 24, 32, 48, 64]))
        n = int(rng.integers(0, 40))
        lens = [2 * cp * int(rng.integers(0, 6)) for _ in range(n)]
        cu = _bounds(lens)
        T = cu[-1]
        f, b = _gpu_pair(cu, T, cp)
        _assert_route(f, oracle.build_route(cu, T, cp, Z2C))
        _assert_route(b, oracle.build_route(cu, T, cp, C2Z))


def test_movedim_wrapper_and_cache():
    cu = _cu_tensor(_bounds(W.random_lengths(3, 20, 2, 6, 0.0)))
    T = int(cu[-1])
    x = torch.randn(3, T, 8, device="cuda").to(torch.bfloat16)   # sequence on dim 1
    cache = thd.RouteCache()
    y = thd.zigzag_contiguous_thd_swap(x, cu, 2, thd.ZIGZAG_TO_CONTIGUOUS, seq_dim=1, cache=cache)
    z = thd.zigzag_contiguous_thd_swap(y, cu, 2, thd.CONTIGUOUS_TO_ZIGZAG, seq_dim=1, cache=cache)
    assert torch.equal(z, x)
    o = oracle.build_route(cu.cpu().tolist(), T, 2, Z2C)
    assert torch.equal(y, x[:, torch.tensor(o.src_of_dst, device="cuda").long()])
    r1 = cache.get(cu, T, 2, thd.ZIGZAG_TO_CONTIGUOUS)
    assert cache.get(cu, T, 2, thd.ZIGZAG_TO_CONTIGUOUS) is r1          # same object: hit
    assert cache.get(cu, T, 2, thd.CONTIGUOUS_TO_ZIGZAG) is not r1      # directions apart
    cu.add_(0)                                                          # in-place write bumps _version
    assert cache.get(cu, T, 2, thd.ZIGZAG_TO_CONTIGUOUS) is not r1
    assert cache.get(cu.clone(), T, 2, thd.ZIGZAG_TO_CONTIGUOUS) is not r1
    r2 = cache.get(cu, T, 2, thd.ZIGZAG_TO_CONTIGUOUS)
    assert cache.get(cu, T, 1, thd.ZIGZAG_TO_CONTIGUOUS) is not r2      # dynamic CP: another cp_size rebuilds
    assert cache.get(cu, T, 2, thd.ZIGZAG_TO_CONTIGUOUS) is not r2      # ... and so does switching back
    assert thd.zigzag_contiguous_thd_swap(x, cu, 1, 0, seq_dim=1) is x  # cp == 1: nothing moves
    pre = thd.RouteCache()
    pre.prebuild(cu, T, 2)                                              # both directions, one launch
    f = pre.get(cu, T, 2, thd.ZIGZAG_TO_CONTIGUOUS)
    b = pre.get(cu, T, 2, thd.CONTIGUOUS_TO_ZIGZAG)
    assert f.src_of_dst.cpu().tolist() == o.src_of_dst
    pre.prebuild(cu, T, 2)                                              # still fresh: nothing rebuilt
    assert pre.get(cu, T, 2, thd.ZIGZAG_TO_CONTIGUOUS) is f and pre.get(cu, T, 2, 1) is b
    assert thd.RouteCache().prebuild(cu, T, 1) is None                  # cp == 1: nothing to build


# --------------------------------------------------------------------------
# labels and packing
# --------------------------------------------------------------------------

@pytest.mark.parametrize("depth", [0, 1, 3])
def test_roll_labels_parity(depth):
    rng = np.random.default_rng(40 + depth)
    for trial in range(12):
        n = int(rng.integers(0, 60))
        lv = [int(rng.integers(0, 40)) for _ in range(n)]
        lp = [L + int(rng.integers(0, 17)) for L in lv]
        cu_v, cu = _bounds(lv), _bounds(lp)
        T = cu[-1]
        tokens = [int(t) for t in rng.integers(0, 151936, size=T)]
        want = oracle.roll_labels(tokens, cu_v, cu, depth, fill=-100)
        st = thd.new_status()
        got = thd.roll_labels(torch.tensor(tokens, dtype=torch.int32, device="cuda"), _cu_tensor(cu_v),
                              _cu_tensor(cu), depth, -100, status=st)
        thd.check_status(st)
        assert got[0].cpu().tolist() == want[0]
        assert got[1].cpu().tolist() == want[1]
        assert got[2].cpu().tolist() == want[2]


@pytest.mark.parametrize("cp,depth", [(1, 0), (2, 1), (3, 1), (4, 3), (6, 0), (8, 2), (16, 3), (64, 1)])
def test_roll_labels_zigzag_parity(cp, depth):
    rng = np.random.default_rng(70 + cp)
    for trial in range(8):
        n = int(rng.integers(0, 80))
        lp = [2 * cp * int(rng.integers(0, 12)) for _ in range(n)]
        lv = [min(L, int(rng.integers(0, L + 3))) if L else 0 for L in lp]
        cu_v, cu = _bounds(lv), _bounds(lp)
        T = cu[-1]
        tokens = [int(t) for t in rng.integers(0, 151936, size=T)]
        want = oracle.roll_labels_zigzag(tokens, cu_v, cu, cp, depth, fill=-7)
        st = thd.new_status()
        got = thd.roll_labels_zigzag(torch.tensor(tokens, dtype=torch.int32, device="cuda"), _cu_tensor(cu_v),
                                     _cu_tensor(cu), cp, depth, -7, status=st)
        thd.check_status(st)
        assert got[0].cpu().tolist() == want[0]
        assert got[1].cpu().tolist() == want[1]
        assert got[2].cpu().tolist() == want[2]


@pytest.mark.parametrize("cp,depth", [(2, 7), (3, 7), (8, 9), (4, 12)])
def test_labels_deep_mtp_both_layouts(cp, depth):
    """MTP depths at and past the seven that the label kernels' token window
    holds (then they read each depth's tokens on their own), with extra
    tokens, in both layouts, against the oracle."""
    rng = np.random.default_rng(900 + 10 * cp + depth)
    for trial in range(6):
        n = int(rng.integers(1, 60))
        lp = [2 * cp * int(rng.integers(0, 14)) for _ in range(n)]
        lv = [min(L, int(rng.integers(0, L + 3))) if L else 0 for L in lp]
        cu_v, cu = _bounds(lv), _bounds(lp)
        T = cu[-1]
        tokens = [int(t) for t in rng.integers(0, 151936, size=T)]
        nxt = [int(rng.integers(200000, 300000)) if (L and rng.random() < 0.4) else None for L in lv]
        nt = torch.tensor([v or 0 for v in nxt], dtype=torch.int32, device="cuda")
        hn = torch.tensor([int(v is not None) for v in nxt], dtype=torch.uint8, device="cuda")
        tok = torch.tensor(tokens, dtype=torch.int32, device="cuda")
        st = thd.new_status()
        got = thd.roll_labels(tok, _cu_tensor(cu_v), _cu_tensor(cu), depth, -9, status=st, next_token=nt,
                              has_next=hn)
        got_z = thd.roll_labels_zigzag(tok, _cu_tensor(cu_v), _cu_tensor(cu), cp, depth, -9, status=st,
                                       next_token=nt, has_next=hn)
        thd.check_status(st)
        assert [g.cpu().tolist() for g in got] == [list(w) for w in oracle.roll_labels(tokens, cu_v, cu, depth,
                                                                                      fill=-9, doc_next=nxt)]
        assert [g.cpu().tolist() for g in got_z] == [list(w) for w in oracle.roll_labels_zigzag(
            tokens, cu_v, cu, cp, depth, fill=-9, doc_next=nxt)]


@pytest.mark.parametrize("cp,n", [(1, 13000), (4, 13000), (4, 24000)])
def test_labels_and_partition_beyond_shared_memory(cp, n):
    """Many documents (empty ones included): with 13,000 the label kernels
    stage both boundary arrays (104 KB) in shared memory above the default
    48 KB and the partition kernel searches global memory; with 24,000 (192
    KB) the label kernels search global memory too.  Labels with MTP depth 2
    and per-document extra tokens, in both layouts, and the partition of
    every rank, against the oracle."""
    rng = np.random.default_rng(123 + cp + n)
    lp = [2 * cp * int(rng.integers(0, 4)) for _ in range(n)]
    lv = [min(L, int(rng.integers(0, L + 3))) if L else 0 for L in lp]
    cu_v, cu = _bounds(lv), _bounds(lp)
    T = cu[-1]
    tokens = [int(t) for t in rng.integers(0, 151936, size=T)]
    nxt = [int(rng.integers(200000, 300000)) if (L and rng.random() < 0.3) else None for L in lv]
    nt = torch.tensor([v or 0 for v in nxt], dtype=torch.int32, device="cuda")
    hn = torch.tensor([int(v is not None) for v in nxt], dtype=torch.uint8, device="cuda")
    tok = torch.tensor(tokens, dtype=torch.int32, device="cuda")
    st = thd.new_status()
    got = thd.roll_labels(tok, _cu_tensor(cu_v), _cu_tensor(cu), 2, -5, status=st, next_token=nt, has_next=hn)
    got_z = thd.roll_labels_zigzag(tok, _cu_tensor(cu_v), _cu_tensor(cu), cp, 2, -5, status=st, next_token=nt,
                                   has_next=hn)
    part = thd.partition_indices(_cu_tensor(cu), T, cp, -1, status=st)
    one = thd.partition_indices(_cu_tensor(cu), T, cp, cp - 1, status=st)
    thd.check_status(st)
    want = oracle.roll_labels(tokens, cu_v, cu, 2, fill=-5, doc_next=nxt)
    assert [g.cpu().tolist() for g in got] == [list(w) for w in want]
    want_z = oracle.roll_labels_zigzag(tokens, cu_v, cu, cp, 2, fill=-5, doc_next=nxt)
    assert [g.cpu().tolist() for g in got_z] == [list(w) for w in want_z]
    assert part.reshape(-1).cpu().tolist() == oracle.partition_indices(cu, T, cp, -1)
    assert one.cpu().tolist() == oracle.partition_indices(cu, T, cp, cp - 1)


def test_extra_tokens_pack_and_labels():
    """Rows with one extra token each: packing reports which documents it
    continues, and both label kernels take it as the target one past the
    document's end."""
    rng = np.random.default_rng(31)
    for trial in range(6):
        B, S = int(rng.integers(1, 6)), int(rng.integers(1, 6000))
        raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
        raw[rng.random((B, S)) < float(rng.choice([0.001, 0.05]))] = 7
        if trial % 2:
            raw[0, -1] = 7                      # a row ending exactly at EOD
        extra = rng.integers(100, 200, size=B).astype(np.int32)
        trim = trial % 3 == 0
        if trim:
            raw[-1, S // 2:] = 0                # trailing pad: no continuation for that row
        align, cp = 8, 4
        tok_o, cu_v_o, cu_o, nxt_o = oracle.pack_docs(raw.tolist(), 7, align, pad_id=0,
                                                       raw_pad_id=0 if trim else None, row_next=extra.tolist())
        tok, cu_v, cu, nt, hn = thd.pack_docs(torch.from_numpy(raw).cuda(), 7, align, pad_id=0,
                                              raw_pad_id=0 if trim else None,
                                              row_next=torch.from_numpy(extra).cuda())
        assert tok.cpu().tolist() == tok_o and cu.cpu().tolist() == cu_o and cu_v.cpu().tolist() == cu_v_o
        assert hn.cpu().tolist() == [int(v is not None) for v in nxt_o]
        assert [v for v, h in zip(nt.cpu().tolist(), hn.cpu().tolist()) if h] == [v for v in nxt_o if v is not None]
        for depth in (0, 2):
            want = oracle.roll_labels(tok_o, cu_v_o, cu_o, depth, fill=-3, doc_next=nxt_o)
            got = thd.roll_labels(tok, cu_v, cu, depth, -3, next_token=nt, has_next=hn)
            assert [g.cpu().tolist() for g in got] == [list(w) for w in want]
            want_z = oracle.roll_labels_zigzag(tok_o, cu_v_o, cu_o, cp, depth, fill=-3, doc_next=nxt_o)
            got_z = thd.roll_labels_zigzag(tok, cu_v, cu, cp, depth, -3, next_token=nt, has_next=hn)
            assert [g.cpu().tolist() for g in got_z] == [list(w) for w in want_z]


def test_pack_docs_worked_example_and_corners():
    E = 99
    cases = [
        ([[1, 2, 3, E, 4, 5, E, 0], [6, 7, 8, 9, 10, E, 0, 0]], 4, 0),
        ([[0, 0, 0, 0], [1, 2, E, 3], [1, 2, 3, E], [E, E, 5, 6], [7, 8, 9, 9], [4, 0, E, 0]], 4, 0),
        ([[0, 0, 0]], 4, 0),
    ]
    for raw, align, rp in cases:
        want = oracle.pack_docs(raw, E, align, pad_id=77, raw_pad_id=rp)
        got = thd.pack_docs(torch.tensor(raw, dtype=torch.int32, device="cuda"), E, align, pad_id=77,
                            raw_pad_id=rp)
        assert [g.cpu().tolist() for g in got] == [list(w) for w in want]


def test_pack_docs_random_against_oracle():
    rng = np.random.default_rng(8)
    for trial in range(10):
        B, S = int(rng.integers(1, 6)), int(rng.integers(1, 20000))
        raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
        raw[rng.random((B, S)) < float(rng.choice([0.0005, 0.01, 0.3]))] = 7
        align = int(rng.choice([1, 4, 16]))
        want = oracle.pack_docs(raw.tolist(), 7, align, pad_id=0)
        got = thd.pack_docs(torch.from_numpy(raw).cuda(), 7, align, pad_id=0)
        assert [g.cpu().tolist() for g in got] == [list(w) for w in want]


def test_pack_docs_long_rows_with_trailing_pad():
    """Rows of several 2048-token chunks whose valid region ends inside a later
    chunk (trailing pads trimmed), documents crossing chunk boundaries."""
    rng = np.random.default_rng(12)
    B, S = 4, 9000
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 0.002] = 7
    ends = [9000, 2049, 6143, 0]                  # last row all pad
    for b, e in enumerate(ends):
        raw[b, e:] = 0
    raw[1, 2048] = 7                              # an EOD exactly at a chunk start
    want = oracle.pack_docs(raw.tolist(), 7, 16, pad_id=5, raw_pad_id=0)
    got = thd.pack_docs(torch.from_numpy(raw).cuda(), 7, 16, pad_id=5, raw_pad_id=0)
    assert [g.cpu().tolist() for g in got] == [list(w) for w in want]


def test_pack_docs_many_chunks_and_rows():
    """More than 1024 chunks and more than 1024 rows: the scan over the chunk
    statistics and over the rows' valid lengths runs in several passes.
    Two rows of just over 2^20 tokens (1026 chunks of 2048), then 1500 short
    rows with trailing pads trimmed and extra tokens."""
    rng = np.random.default_rng(77)
    B, S = 2, 2**20 + 123
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 1 / 3000] = 7
    raw[0, 2048 * 300] = 7                        # an EOD at a chunk start
    want = oracle.pack_docs(raw.tolist(), 7, 8, pad_id=3)
    got = thd.pack_docs(torch.from_numpy(raw).cuda(), 7, 8, pad_id=3)
    assert [g.cpu().tolist() for g in got] == [list(w) for w in want]

    B, S = 1500, 37
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 0.1] = 7
    for b in range(0, B, 3):
        raw[b, int(rng.integers(0, S + 1)):] = 0   # trailing pad (some rows all pad)
    extra = rng.integers(100, 200, size=B).astype(np.int32)
    want = oracle.pack_docs(raw.tolist(), 7, 4, pad_id=0, raw_pad_id=0, row_next=extra.tolist())
    tok, cu_v, cu, nt, hn = thd.pack_docs(torch.from_numpy(raw).cuda(), 7, 4, pad_id=0, raw_pad_id=0,
                                          row_next=torch.from_numpy(extra).cuda())
    assert tok.cpu().tolist() == want[0] and cu_v.cpu().tolist() == want[1] and cu.cpu().tolist() == want[2]
    assert hn.cpu().tolist() == [int(v is not None) for v in want[3]]
    assert [v for v, h in zip(nt.cpu().tolist(), hn.cpu().tolist()) if h] == [v for v in want[3] if v is not None]


# --------------------------------------------------------------------------
# the full-size workloads, in the launch configuration the benchmark times
# --------------------------------------------------------------------------

def _full_size_swap_check(cu, cp, hidden, seed):
    """Both routes exactly, then every row of both directions' payloads
    against the oracle's permutation (target row q = source row
    src_of_dst[q], the oracle's pack -> all-to-all -> scatter composed; the
    oracle tests pin the two to each other), and the round trip."""
    T = cu[-1]
    x = W.payload_device(seed, T, hidden, "cuda")
    pair = _gpu_pair(cu, T, cp)
    outs = {}
    for d in (Z2C, C2Z):
        o = oracle.build_route(cu, T, cp, d)
        r = _gpu_route(cu, T, cp, d)
        _assert_route(r, o)
        _assert_route(pair[d], o)
        st = thd.new_status()
        src = x if d == Z2C else outs[Z2C]
        out = thd.swap(src, r, status=st)
        thd.check_status(st)
        perm = torch.tensor(o.src_of_dst, dtype=torch.int64, device="cuda")
        assert torch.equal(out, src[perm]), f"direction {d}: a row differs from the oracle's"
        del perm
        outs[d] = out
    assert torch.equal(outs[C2Z], x)


@pytest.mark.parametrize("name", ["lognorm128k", "longtail128k", "stress16"])
def test_full_size_workloads(name):
    w = W.BY_NAME[name]
    cu = _bounds(W.doc_lengths(name))
    _full_size_swap_check(cu, w.cp, w.hidden, w.seed)


@pytest.mark.parametrize("name", ["lognorm128k", "longtail128k", "stress16"])
def test_full_size_ulysses(name, chunk=65536):
    """The Ulysses exchange of the full hidden states, every token against the
    oracle (in chunks of tokens, each a sequence of its own for the oracle:
    the exchange moves every token's pieces independently), head -> sequence
    by the round trip.  stress16 splits 512-byte rows 16 ways (32-byte
    pieces, the tile transpose); the 128K workloads have 1 KiB pieces (the
    bulk row engine)."""
    w = W.BY_NAME[name]
    T = sum(W.doc_lengths(name))
    x = W.payload_device(w.seed, T, w.hidden, "cuda")
    heads = x.shape[1]
    st = thd.new_status()
    y = thd.ulysses_swap(x, w.cp, thd.SEQ_TO_HEAD, status=st)
    back = thd.ulysses_swap(y, w.cp, thd.HEAD_TO_SEQ, status=st)
    thd.check_status(st)
    assert y.shape[2] == heads // w.cp
    assert chunk % w.cp == 0 and T % w.cp == 0
    for lo in range(0, T, chunk):
        hi = min(T, lo + chunk)
        xs = x[lo:hi].contiguous().view(torch.uint8).reshape(hi - lo, -1).cpu().numpy()
        want = oracle.ulysses_swap(xs, w.cp, oracle.SEQ_TO_HEAD).reshape(w.cp, hi - lo, -1)
        got = y[:, lo:hi].contiguous().view(torch.uint8).reshape(w.cp, hi - lo, -1).cpu().numpy()
        assert np.array_equal(got, want), f"tokens [{lo}, {hi})"
    assert torch.equal(back, x)


def test_full_size_pipeline():
    w = W.BY_NAME["pipeline"]
    raw = W.raw_pipeline_tokens(w.seed)
    tok_o, cu_v_o, cu_o = oracle.pack_docs(raw.tolist(), W.EOD_ID, 2 * w.cp, pad_id=0)
    tok, cu_v, cu = thd.pack_docs(torch.from_numpy(raw).cuda(), W.EOD_ID, 2 * w.cp, pad_id=0)
    assert tok.cpu().tolist() == tok_o
    assert cu_v.cpu().tolist() == cu_v_o
    assert cu.cpu().tolist() == cu_o
    labels, lmask, valid = thd.roll_labels(tok, cu_v, cu, w.mtp_depth, fill=0)
    lab_o, msk_o, val_o = oracle.roll_labels(tok_o, cu_v_o, cu_o, w.mtp_depth, fill=0)
    assert labels.cpu().tolist() == lab_o
    assert lmask.cpu().tolist() == msk_o
    assert valid.cpu().tolist() == val_o
    # the same labels in the zigzag layout of cp=8 ranks
    zl, zm, zv = thd.roll_labels_zigzag(tok, cu_v, cu, w.cp, w.mtp_depth, fill=0)
    idx = torch.tensor(oracle.partition_indices(cu_o, len(tok_o), w.cp, -1), device="cuda").long()
    assert torch.equal(zl, labels[:, idx]) and torch.equal(zm, lmask[:, idx]) and torch.equal(zv, valid[idx])
    _full_size_swap_check(cu_o, w.cp, w.hidden, w.seed)


def test_pipeline_fuzz():
    """Random raw batches through the whole path, every stage against the
    oracle: packing (EOD density, trailing raw pad, extra tokens), labels and
    MTP targets in both layouts, the partition of every rank, both routes in
    one launch, then the payload swapped there and back for several row
    widths (4, 16, 48, 512 and 4096 bytes: the unit, run and bulk engines)
    and through the three separate steps."""
    rng = np.random.default_rng(2024)
    E = 7
    for trial in range(10):
        cp = int(rng.choice([1, 2, 3, 4, 8]))
        B, S = int(rng.integers(1, 7)), int(rng.integers(1, 2500))
        raw = rng.integers(10, 1000, size=(B, S)).astype(np.int32)
        raw[rng.random((B, S)) < float(rng.choice([0.0005, 0.003, 0.03]))] = E
        trim = trial % 3 == 1
        if trim:
            raw[rng.integers(0, B), S - S // 3:] = 0
        extra = rng.integers(2000, 3000, size=B).astype(np.int32) if trial % 2 else None
        tok_o, cu_v_o, cu_o, *nx = oracle.pack_docs(raw.tolist(), E, 2 * cp, pad_id=0,
                                                    raw_pad_id=0 if trim else None,
                                                    row_next=None if extra is None else extra.tolist())
        nxt_o = nx[0] if nx else None
        got = thd.pack_docs(torch.from_numpy(raw).cuda(), E, 2 * cp, pad_id=0, raw_pad_id=0 if trim else None,
                            row_next=None if extra is None else torch.from_numpy(extra).cuda())
        tok, cu_v, cu = got[:3]
        nt, hn = (got[3], got[4]) if extra is not None else (None, None)
        assert tok.cpu().tolist() == tok_o and cu_v.cpu().tolist() == cu_v_o and cu.cpu().tolist() == cu_o
        T = len(tok_o)
        depth = int(rng.integers(0, 4))
        st = thd.new_status()
        lab = thd.roll_labels(tok, cu_v, cu, depth, -1, status=st, next_token=nt, has_next=hn)
        lab_z = thd.roll_labels_zigzag(tok, cu_v, cu, cp, depth, -1, status=st, next_token=nt, has_next=hn)
        part = thd.partition_indices(cu, T, cp, -1, status=st)
        fwd, bwd = thd.route_build_pair(cu, T, cp, status=st)
        thd.check_status(st)
        assert [g.cpu().tolist() for g in lab] == [list(v) for v in
                                                   oracle.roll_labels(tok_o, cu_v_o, cu_o, depth, fill=-1,
                                                                      doc_next=nxt_o)]
        assert [g.cpu().tolist() for g in lab_z] == [list(v) for v in
                                                     oracle.roll_labels_zigzag(tok_o, cu_v_o, cu_o, cp, depth,
                                                                               fill=-1, doc_next=nxt_o)]
        assert part.reshape(-1).cpu().tolist() == oracle.partition_indices(cu_o, T, cp, -1)
        want = [oracle.build_route(cu_o, T, cp, d) for d in (Z2C, C2Z)]
        _assert_route(fwd, want[Z2C])
        _assert_route(bwd, want[C2Z])
        for row_bytes in (4, 16, 48, 512, 4096):
            x = torch.from_numpy(rng.integers(0, 256, size=(T, row_bytes), dtype=np.uint8)).cuda()
            y = thd.swap(x, fwd, status=st)
            y3 = thd.scatter(thd.a2a_local(thd.pack(x, fwd, status=st), fwd, status=st), fwd, status=st)
            z = thd.swap(y, bwd, status=st)
            thd.check_status(st)
            _, _, y_o = oracle.apply_route(x.cpu().numpy(), want[Z2C])
            assert np.array_equal(y.cpu().numpy(), y_o), (trial, cp, T, row_bytes)
            assert torch.equal(y3, y), (trial, cp, T, row_bytes)
            assert torch.equal(z, x), (trial, cp, T, row_bytes)
