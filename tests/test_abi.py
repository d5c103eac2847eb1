"""The C ABI without a GPU: libthd.so loads, exports every function
include/thd.h declares, and its host-side checks answer without touching a
device (no compute call is made here)."""

import ctypes
import os
import re

import pytest

from context_packed_sequence_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "thd.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(thd_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from context_packed_sequence_gb300 import build
        build.build()
    return L.load()


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = _declared()
    assert len(names) >= 16
    for name in names:
        assert hasattr(lib, name), name
        assert name in L.SIGNATURES, f"{name} has no ctypes signature"
    assert sorted(L.SIGNATURES) == names


def _declarations():
    """(name, return type, [parameter types]) of every function in thd.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = []
    for m in re.finditer(r"([A-Za-z_][\w \*]*?)\b(thd_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        types = []
        if params and params != "void":
            for p in params.split(","):
                p = " ".join(p.split())
                types.append(re.sub(r"\s*\b[A-Za-z_]\w*$", "", p) if not p.endswith("*") else p)
        out.append((name, ret, types))
    return out


def _ctype_for(c_type, is_return=False):
    import ctypes as C
    t = " ".join(c_type.replace("*", " * ").split())
    if t.endswith("*"):
        base = t[:-1].replace("const", "").strip()
        if base == "thd_route_t":
            return ("pointer", "ThdRoute")
        if base == "char":
            return C.c_char_p
        if base == "int32_t" and not is_return:
            return ("pointer", "c_int32_or_void")
        return C.c_void_p
    base = t.replace("const", "").strip()
    return {"int64_t": C.c_int64, "int32_t": C.c_int32, "size_t": C.c_size_t, "thd_status_t": C.c_int32,
            "thd_dir_t": C.c_int32, "thd_ulysses_dir_t": C.c_int32, "cudaStream_t": C.c_void_p}[base]


def test_ctypes_signatures_match_the_header_parameter_by_parameter():
    import ctypes as C
    decls = _declarations()
    assert sorted(d[0] for d in decls) == sorted(L.SIGNATURES)
    for name, ret, params in decls:
        res, args = L.SIGNATURES[name]
        assert res is _ctype_for(ret, is_return=True), (name, ret, res)
        assert len(args) == len(params), (name, params, args)
        for i, (p, a) in enumerate(zip(params, args)):
            want = _ctype_for(p)
            if want == ("pointer", "ThdRoute"):
                assert a is C.POINTER(L.ThdRoute), (name, i, p, a)
            elif want == ("pointer", "c_int32_or_void"):
                assert a in (C.c_void_p, C.POINTER(C.c_int32)), (name, i, p, a)
            else:
                assert a is want, (name, i, p, a)


def test_status_codes_match_header(lib):
    text = open(HEADER).read()
    codes = dict((k, int(v)) for k, v in re.findall(r"THD_(OK|ERR_[A-Z_]+)\s*=\s*(\d+)", text))
    assert codes["OK"] == L.OK
    for name, val in codes.items():
        if name != "OK":
            assert getattr(L, name) == val, name
    assert lib.thd_status_string(L.ERR_LEN_NOT_DIVISIBLE).decode().startswith("sequence length not divisible")
    assert lib.thd_version() == 100


def test_route_struct_layout():
    assert ctypes.sizeof(L.ThdRoute) == 16 + 9 * 8
    assert L.ThdRoute.send_rows.offset == 16


def test_route_bytes_and_bind_host_only(lib):
    assert lib.thd_route_bytes(24, 2) > 0
    assert lib.thd_route_bytes(0, 4) > 0          # T = 0 is legal
    assert lib.thd_route_bytes(26, 2) == 0        # T not a multiple of 2cp
    assert lib.thd_route_bytes(64, 0) == 0
    assert lib.thd_route_bytes(256, 65) == 0      # cp above the maximum
    T, cp = 24, 2
    nbytes = lib.thd_route_bytes(T, cp)
    r = L.ThdRoute()
    fake = 1 << 20  # an aligned address; bind only does arithmetic on it
    assert lib.thd_route_bind(ctypes.byref(r), fake, nbytes, T, cp, 0) == L.OK
    assert (r.cp_size, r.dir, r.total_rows) == (cp, 0, T)
    ptrs = [r.send_rows, r.recv_rows, r.src_of_dst, r.input_split_sizes, r.output_split_sizes,
            r.send_offsets, r.recv_offsets, r.send_identity, r.recv_identity]
    assert all(p % 256 == 0 for p in ptrs)
    assert len(set(ptrs)) == len(ptrs)
    assert max(ptrs) < fake + nbytes
    assert lib.thd_route_bind(ctypes.byref(r), fake, nbytes - 1, T, cp, 0) == L.ERR_INVALID_ARG
    assert lib.thd_route_bind(ctypes.byref(r), fake + 16, nbytes, T, cp, 0) == L.ERR_INVALID_ARG
    assert lib.thd_route_bind(ctypes.byref(r), fake, nbytes, T, cp, 7) == L.ERR_BAD_DIRECTION


def test_host_checks_return_before_any_launch(lib):
    r = L.ThdRoute()
    fake = 1 << 20
    lib.thd_route_bind(ctypes.byref(r), fake, lib.thd_route_bytes(24, 2), 24, 2, 0)
    # direction first, then arguments -- the same order as the oracle
    assert lib.thd_route_build(fake, 3, 24, 2, 9, ctypes.byref(r), fake, None) == L.ERR_BAD_DIRECTION
    assert lib.thd_route_build(fake, 3, 24, 0, 0, ctypes.byref(r), fake, None) == L.ERR_INVALID_ARG
    assert lib.thd_route_build(fake, 3, 26, 2, 0, ctypes.byref(r), fake, None) == L.ERR_INVALID_ARG
    assert lib.thd_route_build(None, 3, 24, 2, 0, ctypes.byref(r), fake, None) == L.ERR_INVALID_ARG
    assert lib.thd_route_build(fake, 3, 24, 2, 0, ctypes.byref(r), None, None) == L.ERR_INVALID_ARG
    # route bound for the other direction / size
    assert lib.thd_route_build(fake, 3, 24, 2, 1, ctypes.byref(r), fake, None) == L.ERR_INVALID_ARG
    assert lib.thd_partition_indices(fake, 3, 24, 2, 2, fake, fake, None) == L.ERR_INVALID_ARG
    assert lib.thd_swap(fake, fake + 8, 16, ctypes.byref(r), None, None) == L.ERR_INVALID_ARG  # overlap
    assert lib.thd_swap(fake, fake + 4096, 0, ctypes.byref(r), None, None) == L.ERR_INVALID_ARG
    assert lib.thd_swap(fake, fake + 4096, 16, None, None, None) == L.ERR_INVALID_ARG
    assert lib.thd_roll_labels(fake, fake, fake, 3, 24, -1, 0, None, None, fake, fake, fake, fake,
                               None) == L.ERR_INVALID_ARG   # depth -1
    assert lib.thd_roll_labels(fake, fake, fake, 3, 24, 0, 0, fake, None, fake, fake, fake, fake,
                               None) == L.ERR_INVALID_ARG   # next_token without has_next
    assert lib.thd_pack_docs(fake, 2, 8, 99, 0, 0, 0, 0, None, fake, 16, fake, fake, None, None, 4, fake, fake,
                             64, fake, None) == L.ERR_INVALID_ARG   # align 0
    assert lib.thd_pack_docs(fake, 2, 8, 99, 0, 0, 4, 0, fake, fake, 16, fake, fake, None, None, 4, fake, fake,
                             64, fake, None) == L.ERR_INVALID_ARG   # row_next without has_next
    # two int64 per row, seven per 2048-token chunk (8 rows x 2 chunks), two totals
    assert lib.thd_pack_docs_workspace_bytes(8, 4096) == 8 * (2 * 8 + 7 * 16 + 2)
    assert lib.thd_status_clear(None, None) == L.ERR_INVALID_ARG


def test_route_pair_bind_host_only(lib):
    """thd_route_bind_pair: one buffer, the shared arrays aliased between the
    two routes, every array 256-byte aligned and inside the buffer."""
    T, cp = 48, 4
    nbytes = lib.thd_route_pair_bytes(T, cp)
    assert nbytes > 0 and nbytes < 2 * lib.thd_route_bytes(T, cp)
    assert lib.thd_route_pair_bytes(50, 4) == 0
    zc, cz = L.ThdRoute(), L.ThdRoute()
    fake = 1 << 20
    assert lib.thd_route_bind_pair(ctypes.byref(zc), ctypes.byref(cz), fake, nbytes, T, cp) == L.OK
    assert (zc.dir, cz.dir) == (0, 1) and zc.total_rows == cz.total_rows == T
    assert zc.recv_rows == cz.send_rows and zc.send_rows == cz.recv_rows
    assert zc.src_of_dst != cz.src_of_dst
    ptrs = []
    for r in (zc, cz):
        ptrs += [r.send_rows, r.recv_rows, r.src_of_dst, r.input_split_sizes, r.output_split_sizes,
                 r.send_offsets, r.recv_offsets, r.send_identity, r.recv_identity]
    assert all(p % 256 == 0 and fake <= p < fake + nbytes for p in ptrs)
    assert len(set(ptrs)) == len(ptrs) - 2          # exactly the two shared arrays repeat
    assert lib.thd_route_bind_pair(ctypes.byref(zc), ctypes.byref(cz), fake, nbytes - 1, T, cp) == L.ERR_INVALID_ARG
    assert lib.thd_route_bind_pair(ctypes.byref(zc), ctypes.byref(cz), fake + 8, nbytes, T, cp) == L.ERR_INVALID_ARG
    assert lib.thd_route_bind_pair(ctypes.byref(zc), ctypes.byref(zc), fake, nbytes, T, cp) == L.ERR_INVALID_ARG
    assert lib.thd_route_bind_pair(None, ctypes.byref(cz), fake, nbytes, T, cp) == L.ERR_INVALID_ARG


def test_batched_and_per_rank_host_checks(lib):
    """thd_swap_batched, thd_pack_rank and thd_scatter_rank refuse bad
    arguments before any launch."""
    T, cp = 24, 2
    r = L.ThdRoute()
    fake = 1 << 20
    lib.thd_route_bind(ctypes.byref(r), fake, lib.thd_route_bytes(T, cp), T, cp, 0)
    big = 1 << 32
    assert lib.thd_swap_batched(big, big + 3 * T * 16 - 16, 3, 16, ctypes.byref(r), None, None) == L.ERR_INVALID_ARG
    assert lib.thd_swap_batched(big, big + 4096, -1, 16, ctypes.byref(r), None, None) == L.ERR_INVALID_ARG
    assert lib.thd_swap_batched(big, big + 4096, (1 << 31) // T + 1, 4, ctypes.byref(r), None,
                                None) == L.ERR_INVALID_ARG                      # outer * T above 2^31 - 1
    assert lib.thd_swap_batched(big, big + 4096, 2, 0, ctypes.byref(r), None, None) == L.ERR_INVALID_ARG
    assert lib.thd_swap_batched(big, big + 4096, 2, 16, None, None, None) == L.ERR_INVALID_ARG
    assert lib.thd_swap_batched(None, None, 0, 16, ctypes.byref(r), None, None) == L.OK   # nothing to move
    S = T // cp
    for fn in (lib.thd_pack_rank, lib.thd_scatter_rank):
        assert fn(big, big + S * 16, cp, 16, ctypes.byref(r), None, None) == L.ERR_INVALID_ARG   # rank >= cp
        assert fn(big, big + S * 16, -1, 16, ctypes.byref(r), None, None) == L.ERR_INVALID_ARG
        assert fn(big, big + 8, 0, 16, ctypes.byref(r), None, None) == L.ERR_INVALID_ARG         # overlap
        assert fn(big, None, 0, 16, ctypes.byref(r), None, None) == L.ERR_INVALID_ARG
        assert fn(big, big + 4096, 0, 16, None, None, None) == L.ERR_INVALID_ARG
