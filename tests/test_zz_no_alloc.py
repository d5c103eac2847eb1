"""thd_pack_docs_noalloc -- packing for callers that cannot allocate device
memory -- against thd_pack_docs, through the C ABI.

Some callers are handed only their input and output buffers (their host
framework's pool owns the rest of device memory) or must not call
cudaMalloc/cudaFree, which can synchronise the device.  The no-allocation
entry point serves them from a fixed scratch array inside the library.  Its
results must equal thd_pack_docs's exactly (integer outputs, tolerance 0), on
consecutive calls that share that scratch, and a batch larger than the
scratch must be refused before anything is enqueued.
"""

import ctypes

import numpy as np
import pytest
import torch

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
    return tok[:T].cpu().tolist(), cu_v[:n + 1].cpu().tolist(), cu[:n + 1].cpu().tolist(), (n, T)


def _with_workspace(lib, raw, eod, align, pad_id, trim, raw_pad):
    B, S = raw.shape
    tok, cu_v, cu, counts, st = _outputs(B, S, align, raw.device)
    ws = torch.empty(max(lib.thd_pack_docs_workspace_bytes(B, S), 8), dtype=torch.uint8, device=raw.device)
    code = lib.thd_pack_docs(raw.data_ptr(), B, S, eod, trim, raw_pad, align, pad_id, None, tok.data_ptr(),
                             tok.numel(), cu_v.data_ptr(), cu.data_ptr(), None, None, cu.numel(), counts.data_ptr(),
                             ws.data_ptr(), ws.numel(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == L.OK
    return _result(tok, cu_v, cu, counts, st)


def _no_alloc(lib, raw, eod, align, pad_id, trim, raw_pad):
    B, S = raw.shape
    tok, cu_v, cu, counts, st = _outputs(B, S, align, raw.device)
    code = lib.thd_pack_docs_noalloc(raw.data_ptr(), B, S, eod, trim, raw_pad, align, pad_id, tok.data_ptr(),
                                     tok.numel(), cu_v.data_ptr(), cu.data_ptr(), cu.numel(), counts.data_ptr(),
                                     st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == L.OK
    return _result(tok, cu_v, cu, counts, st)


def test_no_alloc_matches_workspace_entry_point_on_consecutive_calls():
    lib = L.load()
    dev = torch.device("cuda")
    big = torch.from_numpy(W.raw_pipeline_tokens(W.SEED + 4)).to(dev)          # [8, 32768], EOD gaps ~2048
    E = 99
    small = torch.tensor([[1, 2, 3, E, 4, 5, E, 0], [6, 7, 8, 9, 10, E, 0, 0], [0, 0, 0, 0, 0, 0, 0, 0]],
                         dtype=torch.int32, device=dev)
    calls = [
        (big, W.EOD_ID, 16, 0, 0, 0),      # the 8 x 32768 pipeline rows, cp=8 alignment
        (small, E, 4, 77, 1, 0),           # fewer rows than the call before: old scratch must not leak
        (big, W.EOD_ID, 16, 0, 0, 0),      # and the first input again
    ]
    for raw, eod, align, pad_id, trim, raw_pad in calls:
        want = _with_workspace(lib, raw, eod, align, pad_id, trim, raw_pad)
        got = _no_alloc(lib, raw, eod, align, pad_id, trim, raw_pad)
        assert got == want


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
