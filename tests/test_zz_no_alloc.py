"""thd_pack_docs_noalloc -- packing for callers that cannot allocate device
memory -- against the CPU oracle and against thd_pack_docs, through the C ABI.

Some callers are handed only their input and output buffers (their host
framework's pool owns the rest of device memory) or must not call
cudaMalloc/cudaFree, which can synchronise the device.  The no-allocation
entry point serves them from a fixed scratch array inside the library.  Its
results must equal the oracle's and thd_pack_docs's exactly (integer outputs,
tolerance 0), on consecutive calls that share that scratch, at the edges of
the array (no rows, empty rows, exactly THD_PACK_NOALLOC_MAX_ROWS rows, and
both sides of the 512-row switch to a separate prefix-scan kernel), and a
batch larger than the scratch must be refused before anything is enqueued.
"""

import numpy as np
import pytest
import torch

import oracle
from context_packed_sequence_gb300 import _lib as L
import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(B, S, align, dev):
    cap_tok, cap_docs = max(B * S * align, 1), B * S + 1
    return (torch.full((cap_tok,), -9, dtype=torch.int32, device=dev),
            torch.full((cap_docs,), -9, dtype=torch.int32, device=dev),
            torch.full((cap_docs,), -9, dtype=torch.int32, device=dev),
            torch.zeros(2, dtype=torch.int64, device=dev),
            torch.zeros(1, dtype=torch.int32, device=dev))


def _result(tok, cu_v, cu, counts, status):
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    n, T = (int(v) for v in counts.tolist())
    return tok[:T].cpu().tolist(), cu_v[:n + 1].cpu().tolist(), cu[:n + 1].cpu().tolist()


def _raw_ptr(raw):
    # an empty batch passes no buffer at all
    return raw.data_ptr() if raw.numel() else None


def _with_workspace(lib, raw, eod, align, pad_id, trim, raw_pad):
    B, S = raw.shape
    tok, cu_v, cu, counts, st = _outputs(B, S, align, raw.device)
    ws = torch.empty(max(lib.thd_pack_docs_workspace_bytes(B, S), 8), dtype=torch.uint8, device=raw.device)
    code = lib.thd_pack_docs(_raw_ptr(raw), B, S, eod, trim, raw_pad, align, pad_id, None, tok.data_ptr(),
                             tok.numel(), cu_v.data_ptr(), cu.data_ptr(), None, None, cu.numel(), counts.data_ptr(),
                             ws.data_ptr(), ws.numel(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == L.OK
    return _result(tok, cu_v, cu, counts, st)


def _no_alloc(lib, raw, eod, align, pad_id, trim, raw_pad):
    B, S = raw.shape
    tok, cu_v, cu, counts, st = _outputs(B, S, align, raw.device)
    code = lib.thd_pack_docs_noalloc(_raw_ptr(raw), B, S, eod, trim, raw_pad, align, pad_id, tok.data_ptr(),
                                     tok.numel(), cu_v.data_ptr(), cu.data_ptr(), cu.numel(), counts.data_ptr(),
                                     st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == L.OK
    return _result(tok, cu_v, cu, counts, st)


def _check(lib, raw_np, eod, align, pad_id, trim, raw_pad, calls=2):
    """The no-allocation call `calls` times in a row against the oracle and
    the workspace entry point."""
    want = oracle.pack_docs(raw_np.tolist(), eod, align, pad_id=pad_id, raw_pad_id=raw_pad if trim else None)
    want = [list(v) for v in want]
    raw = torch.from_numpy(np.ascontiguousarray(raw_np, dtype=np.int32).reshape(raw_np.shape)).cuda()
    assert [list(v) for v in _with_workspace(lib, raw, eod, align, pad_id, trim, raw_pad)] == want
    for _ in range(calls):
        assert [list(v) for v in _no_alloc(lib, raw, eod, align, pad_id, trim, raw_pad)] == want


def _long_trimmed_rows():
    """Rows longer than one 8,192-token tile of the per-row kernels, trailing
    pads trimmed at and around tile boundaries, EODs exactly at the last and
    first token of a tile, documents crossing tiles (one spans three)."""
    rng = np.random.default_rng(31)
    B, S = 5, 20000
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 0.0004] = 7
    raw[0, 8191] = 7
    raw[0, 8192] = 7
    raw[2, 16383] = 7
    raw[3, :] = np.where(raw[3, :] == 7, 8, raw[3, :])   # no EOD: one document of 17,001 tokens
    for b, e in enumerate([20000, 8193, 16384, 17001, 8192]):
        raw[b, e:] = 0
    return raw


def test_no_alloc_matches_oracle_and_workspace_entry_point_on_consecutive_calls():
    lib = L.load()
    E = 99
    small = np.array([[1, 2, 3, E, 4, 5, E, 0], [6, 7, 8, 9, 10, E, 0, 0], [0, 0, 0, 0, 0, 0, 0, 0]],
                     dtype=np.int32)
    big = W.raw_pipeline_tokens(W.SEED + 4)                       # [8, 32768], EOD gaps ~2048
    # consecutive calls on one stream share the scratch: a smaller batch after
    # a larger one must not see the larger one's leftovers
    _check(lib, big, W.EOD_ID, 16, 0, 0, 0)
    _check(lib, small, E, 4, 77, 1, 0)
    _check(lib, _long_trimmed_rows(), 7, 16, 5, 1, 0)
    _check(lib, big, W.EOD_ID, 16, 0, 0, 0)


@pytest.mark.parametrize("B", [512, 513, L.PACK_NOALLOC_MAX_ROWS])
def test_no_alloc_many_short_rows(B):
    """Short rows up to the array's row limit, trailing pads trimmed (some rows
    all pad, one row just EODs): both sides of the 512-row switch to the
    separate prefix scan, and exactly THD_PACK_NOALLOC_MAX_ROWS rows."""
    lib = L.load()
    rng = np.random.default_rng(B)
    S = 5
    raw = rng.integers(1, 20, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 0.25] = 3
    for b in range(0, B, 7):
        raw[b, int(rng.integers(0, S + 1)):] = 0
    raw[1, :] = 3
    _check(lib, raw, 3, 8, 9, 1, 0)


@pytest.mark.parametrize("B,S", [(0, 0), (0, 16), (2, 0)])
def test_no_alloc_empty_batches(B, S):
    """No rows at all, and rows of no tokens (the raw pointer may be NULL):
    no documents, T = 0, the boundaries start at 0."""
    lib = L.load()
    raw = np.zeros((B, S), dtype=np.int32)
    for trim in (0, 1):
        _check(lib, raw, 7, 4, 0, trim, 0)


def test_no_alloc_refuses_batches_beyond_its_scratch():
    lib = L.load()
    dev = torch.device("cuda")
    B = L.PACK_NOALLOC_MAX_ROWS + 1
    raw = torch.zeros((B, 4), dtype=torch.int32, device=dev)
    tok, cu_v, cu, counts, st = _outputs(B, 4, 2, dev)
    code = lib.thd_pack_docs_noalloc(raw.data_ptr(), B, 4, 1, 0, 0, 2, 0, tok.data_ptr(), tok.numel(),
                                     cu_v.data_ptr(), cu.data_ptr(), cu.numel(), counts.data_ptr(), st.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert code == L.ERR_SCRATCH_LIMIT
    assert "scratch" in lib.thd_status_string(code).decode()
    torch.cuda.synchronize()
    assert bool((cu[:4] == -9).all()) and int(counts.abs().sum()) == 0 and int(st.item()) == 0


def test_no_alloc_capacity_error_above_the_scan_switch():
    """With the separate prefix scan (more than 512 rows) a too-small output
    is reported by that kernel and nothing but the counts is written."""
    lib = L.load()
    dev = torch.device("cuda")
    B, S = 600, 4
    raw = torch.full((B, S), 5, dtype=torch.int32, device=dev)   # one 4-token document per row
    tok = torch.full((B * S - 1,), -9, dtype=torch.int32, device=dev)
    cu_v = torch.full((B + 1,), -9, dtype=torch.int32, device=dev)
    cu = torch.full((B + 1,), -9, dtype=torch.int32, device=dev)
    counts = torch.zeros(2, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    code = lib.thd_pack_docs_noalloc(raw.data_ptr(), B, S, 7, 0, 0, 4, 0, tok.data_ptr(), tok.numel(),
                                     cu_v.data_ptr(), cu.data_ptr(), cu.numel(), counts.data_ptr(), st.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert code == L.OK
    torch.cuda.synchronize()
    assert int(st.item()) == L.ERR_CAPACITY
    assert counts.tolist() == [B, B * S]
    assert bool((tok == -9).all()) and bool((cu == -9).all()) and bool((cu_v == -9).all())
