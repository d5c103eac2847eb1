"""The largest packings the C ABI accepts: T = 2^31 - 16 rows (row indices are
int32) at cp = 8, and T = 2^31 - 2 at cp = 1, where a rank's slots run up to
the top of the int32 range.

One document of about 2^31 rows comes first (its chunks are ~1.3e8 rows, so
the closed forms run at the top of the int32 range), then a thousand small
documents, empty ones included, whose rows sit just below INT32_MAX.  The
oracle cannot build a route of 2^31 rows, so the whole outputs are checked
through properties that hold at any size, and the small documents through
the oracle on each one as a sub-problem (a document's slots, and its labels,
depend only on that document and where it starts):

- the contiguous -> zigzag permutation equals the partition of every rank,
  and the zigzag -> contiguous one is its inverse;
- every rank's rows ascend; the split sizes add up; identity flags agree with
  the rows they summarise;
- a swap there and back returns the payload, whose rows carry their index;
- labels of the small documents and of the large document's tail equal the
  oracle's on that document;
- at cp = 1 the zigzag layout is the contiguous one (each document's two
  chunks in order), so the partition and both routes are the identity and the
  labels written in the zigzag layout equal the contiguous ones.

About 100 GB of device memory at the peak."""

import numpy as np
import pytest
import torch

import oracle
import context_packed_sequence_gb300 as thd

pytestmark = pytest.mark.gpu

T_MAX = 2**31 - 16
CP = 8


def _packing():
    rng = np.random.default_rng(2**31 - 16)
    tail = 16 * rng.integers(1, 33, size=1000)           # 16 .. 512 rows, multiples of 2cp
    tail[rng.choice(1000, size=20, replace=False)] = 0    # empty documents
    head = T_MAX - int(tail.sum())
    lengths = [head] + tail.tolist()
    valid = [head - 5] + [max(0, int(x) - int(rng.integers(0, 16))) for x in tail]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    cu_v = np.concatenate([[0], np.cumsum(valid)]).astype(np.int64)
    assert cu[-1] == T_MAX and head % (2 * CP) == 0
    return cu.tolist(), cu_v.tolist()


@pytest.fixture(scope="module")
def big_gpu():
    props = torch.cuda.get_device_properties(0)
    if props.total_memory < 160 * 2**30:
        pytest.skip("needs a GPU with at least 160 GiB")
    yield
    torch.cuda.empty_cache()


def _small_docs(cu, count=60):
    idx = [i for i in range(1, len(cu) - 1) if cu[i + 1] > cu[i]]
    pick = np.random.default_rng(7).choice(len(idx), size=count, replace=False)
    return sorted({idx[k] for k in pick} | {idx[-1]})


def test_route_partition_and_swap_at_the_row_limit(big_gpu):
    cu, _ = _packing()
    T, S = T_MAX, T_MAX // CP
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    st = thd.new_status()
    part = thd.partition_indices(cu_d, T, CP, -1, status=st)
    fwd, bwd = thd.route_build_pair(cu_d, T, CP, status=st)
    thd.check_status(st)

    # contiguous -> zigzag: zigzag position u takes global row part[u]
    assert torch.equal(bwd.src_of_dst, part.reshape(-1))
    assert bool((part[:, 1:] > part[:, :-1]).all())
    # the small documents against the oracle, one document at a time
    for i in _small_docs(cu):
        L = cu[i + 1] - cu[i]
        lo, hi = cu[i] // CP, cu[i + 1] // CP
        for r in range(CP):
            want = [cu[i] + v for v in oracle.partition_indices([0, L], L, CP, r)]
            assert part[r, lo:hi].cpu().tolist() == want, (i, r)
    # zigzag -> contiguous is the inverse permutation
    inv = fwd.src_of_dst.index_select(0, part.reshape(-1).long())
    assert torch.equal(inv, torch.arange(T, dtype=torch.int32, device="cuda"))
    del inv

    # split sizes, offsets and identity flags against the rows they describe
    for r in (fwd, bwd):
        assert r.input_split_sizes.sum(1).tolist() == [S] * CP
        assert torch.equal(r.input_split_sizes, r.output_split_sizes.t())
    ar = torch.arange(S, dtype=torch.int32, device="cuda")
    for d in range(CP):
        assert bool(fwd.send_identity[d]) and bool(bwd.recv_identity[d])
        assert bool(fwd.recv_identity[d]) == torch.equal(fwd.recv_rows[d], ar)
        assert bool(bwd.send_identity[d]) == torch.equal(bwd.send_rows[d], ar)
    del ar, part

    # a swap there and back; every row carries its own index
    x = torch.arange(T, dtype=torch.int32, device="cuda").view(T, 1)
    y = thd.swap(x, fwd, status=st)
    assert torch.equal(y.view(-1), fwd.src_of_dst)
    z = thd.swap(y, bwd, status=st)
    thd.check_status(st)
    assert torch.equal(z, x)


def test_labels_at_the_row_limit(big_gpu):
    cu, cu_v = _packing()
    T = T_MAX
    dev = lambda v: torch.tensor(v, dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(31)
    tokens = torch.randint(0, 151643, (T,), dtype=torch.int32, device="cuda", generator=g)
    st = thd.new_status()
    labels, lmask, valid = thd.roll_labels(tokens, dev(cu_v), dev(cu), 1, fill=-1, status=st)
    thd.check_status(st)

    def check(lo, hi, vlen):
        toks = tokens[lo:hi].cpu().tolist()
        want = oracle.roll_labels(toks, [0, vlen], [0, hi - lo], 1, fill=-1)
        assert labels[:, lo:hi].cpu().tolist() == want[0], (lo, hi)
        assert lmask[:, lo:hi].cpu().tolist() == want[1], (lo, hi)
        assert valid[lo:hi].cpu().tolist() == want[2], (lo, hi)

    for i in _small_docs(cu):
        check(cu[i], cu[i + 1], cu_v[i + 1] - cu_v[i])
    # the last 64 rows of the large document: its valid end lies 5 rows
    # before its padded end, and labels only look forward
    head, head_valid = cu[1], cu_v[1]
    check(head - 64, head, 64 - (head - head_valid))
    assert int(valid.sum(dtype=torch.int64)) == cu_v[-1]


T_MAX_CP1 = 2**31 - 2


def _packing_cp1():
    rng = np.random.default_rng(2**31 - 2)
    tail = 2 * rng.integers(1, 257, size=500)              # 2 .. 512 rows, multiples of 2cp = 2
    tail[rng.choice(500, size=10, replace=False)] = 0     # empty documents
    head = T_MAX_CP1 - int(tail.sum())
    lengths = [head] + tail.tolist()
    valid = [head - 3] + [max(0, int(x) - int(rng.integers(0, 2))) for x in tail]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    cu_v = np.concatenate([[0], np.cumsum(valid)]).astype(np.int64)
    assert cu[-1] == T_MAX_CP1 and head % 2 == 0
    return cu.tolist(), cu_v.tolist()


def _is_arange(t, chunk=2**28):
    """t (int32, flat) equals 0, 1, ..., numel-1, compared a chunk at a time."""
    n = t.numel()
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        if not torch.equal(t[lo:hi], torch.arange(lo, hi, dtype=torch.int32, device=t.device)):
            return False
    return True


def test_cp1_partition_and_routes_at_the_row_limit(big_gpu):
    cu, _ = _packing_cp1()
    T = T_MAX_CP1
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    st = thd.new_status()
    part = thd.partition_indices(cu_d, T, 1, -1, status=st)
    thd.check_status(st)
    assert _is_arange(part.reshape(-1))
    part = thd.partition_indices(cu_d, T, 1, 0, status=st, out=part.reshape(-1))
    thd.check_status(st)
    assert _is_arange(part)
    del part
    fwd, bwd = thd.route_build_pair(cu_d, T, 1, status=st)
    thd.check_status(st)
    for r in (fwd, bwd):
        assert _is_arange(r.src_of_dst)
        assert _is_arange(r.send_rows.reshape(-1)) and _is_arange(r.recv_rows.reshape(-1))
        assert r.input_split_sizes.tolist() == [[T]] and r.output_split_sizes.tolist() == [[T]]
        assert bool(r.send_identity[0]) and bool(r.recv_identity[0])


def test_cp1_zigzag_labels_at_the_row_limit(big_gpu):
    cu, cu_v = _packing_cp1()
    T = T_MAX_CP1
    dev = lambda v: torch.tensor(v, dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(37)
    tokens = torch.randint(0, 151643, (T,), dtype=torch.int32, device="cuda", generator=g)
    st = thd.new_status()
    want = thd.roll_labels(tokens, dev(cu_v), dev(cu), 1, fill=-1, status=st)
    got = thd.roll_labels_zigzag(tokens, dev(cu_v), dev(cu), 1, 1, fill=-1, status=st)
    thd.check_status(st)
    for a, b in zip(got, want):
        assert a.shape == b.shape
        for lo in range(0, T, 2**28):
            assert torch.equal(a[..., lo:lo + 2**28], b[..., lo:lo + 2**28]), lo
