"""The single-pass packing (thd_pack_docs from 2^19 raw tokens, 16-byte
aligned rows of a multiple of 4 tokens, 16-byte aligned output): one
persistent kernel whose blocks take 8,192-token chunks in order and look back
over the published summaries of the chunks before them.  Every output is
compared with the oracle's pack_docs ("Packed Sequence 与上下文并行", section
2.2 and the worked example of section 3) element by element: documents
crossing chunk and row boundaries, trimmed rows (some all pad, some ending
exactly at a chunk boundary), extra tokens, many short documents whose padded
output no longer fits the block's shared-memory assembly, alignment 1, rows
shorter than a chunk, and the capacity check."""

import ctypes
import os

import numpy as np
import pytest
import torch

import context_packed_sequence_gb300 as thd
from context_packed_sequence_gb300 import _lib as L
from oracle import thd_oracle as O

pytestmark = pytest.mark.gpu

CHUNK = 8192


def _check(raw, eod, align, pad_id=0, trim=False, extra=None):
    want = O.pack_docs(raw.tolist(), eod, align, pad_id=pad_id, raw_pad_id=0 if trim else None,
                       row_next=None if extra is None else extra.tolist())
    got = thd.pack_docs(torch.from_numpy(raw).cuda(), eod, align, pad_id=pad_id, raw_pad_id=0 if trim else None,
                        row_next=None if extra is None else torch.from_numpy(extra).cuda())
    assert np.array_equal(got[0].cpu().numpy(), np.asarray(want[0], dtype=np.int32))
    assert got[1].cpu().tolist() == want[1]
    assert got[2].cpu().tolist() == want[2]
    if extra is not None:
        hn = got[4].cpu().tolist()
        assert hn == [int(v is not None) for v in want[3]]
        assert [v for v, h in zip(got[3].cpu().tolist(), hn) if h] == [v for v in want[3] if v is not None]


def test_two_long_rows_with_ends_at_chunk_edges():
    rng = np.random.default_rng(301)
    B, S = 2, 2**21 + 8                              # 257 chunks per row, the last one of 8 tokens
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 1 / 3000] = 7
    for k in (1, 2, 3, 100, 255):
        raw[0, k * CHUNK] = 7                          # an EOD at a chunk's first token
        raw[1, k * CHUNK - 1] = 7                      # ... at a chunk's last token
    raw[0, 40 * CHUNK:47 * CHUNK] = 11                 # a document spanning seven chunks
    _check(raw, 7, 8, pad_id=3)


def test_trimmed_rows_and_extra_tokens():
    rng = np.random.default_rng(302)
    B, S = 64, 65536                                   # 8 chunks per row
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 1 / 1500] = 9
    ends = rng.integers(0, S + 1, size=B)
    ends[:8] = [0, S, CHUNK, CHUNK + 1, CHUNK - 1, 3 * CHUNK, 1, 5]  # all pad, full, at / beside a chunk edge
    for b, e in enumerate(ends):
        raw[b, e:] = 0
    raw[5, 2 * CHUNK - 1] = 9
    extra = rng.integers(100, 200, size=B).astype(np.int32)
    _check(raw, 9, 16, pad_id=0, trim=True, extra=extra)


def test_many_short_documents_written_directly():
    """Documents of about 3 tokens padded to 16: a chunk's output is several
    times its input and goes out without the shared-memory assembly."""
    rng = np.random.default_rng(303)
    B, S = 512, 8192
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 0.3] = 7
    raw[::7, -1] = 7
    _check(raw, 7, 16, pad_id=1)


def test_alignment_one_and_mixed_density():
    rng = np.random.default_rng(304)
    B, S = 16, 2**18
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    p = np.where(np.arange(B)[:, None] % 2 == 0, 1 / 20000, 0.05)
    raw[rng.random((B, S)) < p] = 7
    _check(raw, 7, 1)
    _check(raw, 7, 3, pad_id=2)                       # an alignment that is not a power of two


def test_rows_shorter_than_a_chunk():
    rng = np.random.default_rng(305)
    B, S = 4096, 1024
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 1 / 700] = 7
    for b in range(0, B, 5):
        raw[b, int(rng.integers(0, S + 1)):] = 0
    _check(raw, 7, 8, trim=True)


def test_smallest_single_pass_batches():
    """Just above and at the single pass's lower size (2^19 raw tokens): one
    row, and many short rows with trimmed tails and extra tokens."""
    rng = np.random.default_rng(310)
    raw = rng.integers(1, 50, size=(1, 2**19)).astype(np.int32)
    raw[rng.random(raw.shape) < 1 / 1000] = 7
    _check(raw, 7, 16)
    B, S = 128, 4096
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 1 / 300] = 7
    for b in range(0, B, 3):
        raw[b, int(rng.integers(0, S + 1)):] = 0
    _check(raw, 7, 8, trim=True, extra=rng.integers(100, 200, size=B).astype(np.int32))


def test_unaligned_row_length_takes_the_chunked_kernels():
    """S not a multiple of 4 at a single-pass size: the three chunked kernels."""
    rng = np.random.default_rng(306)
    B, S = 2, 2**21 + 7
    raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
    raw[rng.random((B, S)) < 1 / 2500] = 7
    _check(raw, 7, 8)


def test_capacity_on_the_single_pass():
    rng = np.random.default_rng(307)
    raw = rng.integers(1, 50, size=(4, 2**20)).astype(np.int32)
    raw[rng.random(raw.shape) < 1 / 2500] = 99
    want = O.pack_docs(raw.tolist(), 99, 16)
    T, n = len(want[0]), len(want[1]) - 1
    x = torch.from_numpy(raw).cuda()
    with pytest.raises(thd.ThdError) as e:
        thd.pack_docs(x, 99, 16, tokens_capacity=T - 1)
    assert e.value.kind == "capacity"
    tok, cu_v, cu = thd.pack_docs(x, 99, 16, tokens_capacity=T)
    assert np.array_equal(tok.cpu().numpy(), np.asarray(want[0], dtype=np.int32))
    assert cu.cpu().tolist() == want[2] and cu_v.cpu().tolist() == want[1] and len(want[1]) == n + 1


def test_repeated_calls_reuse_the_workspace():
    """Back-to-back calls on one stream: each call clears the flags it uses."""
    rng = np.random.default_rng(308)
    raw = rng.integers(1, 50, size=(8, 2**19)).astype(np.int32)
    raw[rng.random(raw.shape) < 1 / 4000] = 7
    want = O.pack_docs(raw.tolist(), 7, 8)
    x = torch.from_numpy(raw).cuda()
    B, S = raw.shape
    dev = x.device
    tokens = torch.empty(B * S * 8, dtype=torch.int32, device=dev)
    cu_v = torch.empty(B * S + 1, dtype=torch.int32, device=dev)
    cu = torch.empty(B * S + 1, dtype=torch.int32, device=dev)
    counts = torch.zeros(2, dtype=torch.int64, device=dev)
    lib = L.load()
    ws = torch.full((lib.thd_pack_docs_workspace_bytes(B, S),), 0xAB, dtype=torch.uint8, device=dev)
    st = thd.new_status(dev)
    for _ in range(3):
        code = lib.thd_pack_docs(x.data_ptr(), B, S, 7, 0, 0, 8, 0, None, tokens.data_ptr(), tokens.numel(),
                                 cu_v.data_ptr(), cu.data_ptr(), None, None, cu.numel(), counts.data_ptr(),
                                 ws.data_ptr(), ws.numel(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert code == L.OK
    assert thd.status_read(st) == L.OK
    n, T = counts.tolist()
    assert T == len(want[0]) and n == len(want[1]) - 1
    assert np.array_equal(tokens[:T].cpu().numpy(), np.asarray(want[0], dtype=np.int32))
    assert cu[:n + 1].cpu().tolist() == want[2] and cu_v[:n + 1].cpu().tolist() == want[1]


@pytest.mark.skipif(os.environ.get("THD_CHECKED") != "1", reason="the debug request is in the checked build only")
def test_look_back_wait_gives_up_on_a_flag_nobody_sets():
    """The block of chunk 0 publishes nothing: chunk 1's bounded wait runs out,
    the call reports THD_ERR_TIMEOUT and completes, and the next call packs
    normally on the same context."""
    rng = np.random.default_rng(309)
    raw = rng.integers(1, 50, size=(4, 2**20)).astype(np.int32)
    raw[rng.random(raw.shape) < 1 / 2500] = 7
    x = torch.from_numpy(raw).cuda()
    lib = L.load()
    stall = lib.thd_debug_stall_next_pack
    stall.restype, stall.argtypes = ctypes.c_int, [ctypes.c_void_p]
    assert stall(torch.cuda.current_stream().cuda_stream) == L.OK
    with pytest.raises(thd.ThdError) as e:
        thd.pack_docs(x, 7, 8)
    assert e.value.kind == "timeout"
    want = O.pack_docs(raw.tolist(), 7, 8)
    tok, cu_v, cu = thd.pack_docs(x, 7, 8)
    assert np.array_equal(tok.cpu().numpy(), np.asarray(want[0], dtype=np.int32))
    assert cu.cpu().tolist() == want[2]


def _raw_call(lib, x, B, S, outs, ws, st, stream):
    tokens, cu_v, cu, counts = outs
    return lib.thd_pack_docs(x.data_ptr(), B, S, 7, 0, 0, 8, 0, None, tokens.data_ptr(), tokens.numel(),
                             cu_v.data_ptr(), cu.data_ptr(), None, None, cu.numel(), counts.data_ptr(),
                             ws.data_ptr(), ws.numel(), st.data_ptr(), stream.cuda_stream)


def _outputs(B, S, dev):
    return (torch.empty(B * S * 8, dtype=torch.int32, device=dev), torch.empty(B * S + 1, dtype=torch.int32, device=dev),
            torch.empty(B * S + 1, dtype=torch.int32, device=dev), torch.zeros(2, dtype=torch.int64, device=dev))


def _assert_outputs(outs, want):
    tokens, cu_v, cu, counts = outs
    n, T = counts.tolist()
    assert T == len(want[0]) and n == len(want[1]) - 1
    assert np.array_equal(tokens[:T].cpu().numpy(), np.asarray(want[0], dtype=np.int32))
    assert cu[:n + 1].cpu().tolist() == want[2] and cu_v[:n + 1].cpu().tolist() == want[1]


def test_single_pass_in_a_cuda_graph():
    """The single pass captured in a CUDA graph (the clearing kernel and the
    persistent kernel) and replayed three times on changing input: every
    replay clears the counters and records it uses."""
    rng = np.random.default_rng(311)
    B, S = 4, 2**18
    lib = L.load()
    dev = torch.device("cuda")
    x = torch.empty((B, S), dtype=torch.int32, device=dev)
    outs = _outputs(B, S, dev)
    ws = torch.empty(lib.thd_pack_docs_workspace_bytes(B, S), dtype=torch.uint8, device=dev)
    st = thd.new_status(dev)
    side = torch.cuda.Stream()
    x.copy_(torch.from_numpy(rng.integers(1, 50, size=(B, S)).astype(np.int32)))
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one eager call first (loads the kernels into the context)
        assert _raw_call(lib, x, B, S, outs, ws, st, side) == L.OK
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        assert _raw_call(lib, x, B, S, outs, ws, st, torch.cuda.current_stream()) == L.OK
    for trial in range(3):
        raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
        raw[rng.random(raw.shape) < (1 / 500, 1 / 5000, 1 / 50)[trial]] = 7
        x.copy_(torch.from_numpy(raw))
        g.replay()
        torch.cuda.synchronize()
        assert thd.status_read(st) == L.OK
        _assert_outputs(outs, O.pack_docs(raw.tolist(), 7, 8))


def test_two_streams_with_their_own_workspaces():
    """Two single-pass calls that may overlap on the GPU (two streams, no
    ordering between them), each with its own workspace and outputs."""
    rng = np.random.default_rng(312)
    B, S = 4, 2**18
    lib = L.load()
    dev = torch.device("cuda")
    raws = []
    for k in range(2):
        raw = rng.integers(1, 50, size=(B, S)).astype(np.int32)
        raw[rng.random(raw.shape) < (1 / 700, 1 / 3000)[k]] = 7
        raws.append(raw)
    xs = [torch.from_numpy(r).to(dev) for r in raws]
    outs = [_outputs(B, S, dev) for _ in range(2)]
    wss = [torch.empty(lib.thd_pack_docs_workspace_bytes(B, S), dtype=torch.uint8, device=dev) for _ in range(2)]
    sts = [thd.new_status(dev) for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    torch.cuda.synchronize()
    for _ in range(3):
        for k in range(2):
            with torch.cuda.stream(streams[k]):
                assert _raw_call(lib, xs[k], B, S, outs[k], wss[k], sts[k], streams[k]) == L.OK
    torch.cuda.synchronize()
    for k in range(2):
        assert thd.status_read(sts[k]) == L.OK
        _assert_outputs(outs[k], O.pack_docs(raws[k].tolist(), 7, 8))
