"""ctypes declarations of libthd's C ABI (include/thd.h): marshalling only.

Loading fails loudly when the library has not been built; there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_int32, c_int64, c_size_t, c_void_p, c_char_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libthd.so")
# THD_CHECKED=1 in the environment: the debug build, whose kernels range-check
# every row index they compute (built by `build --checked` / build())
CHECKED_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libthd_checked.so")


def lib_path() -> str:
    return CHECKED_LIB_PATH if os.environ.get("THD_CHECKED", "0") == "1" else LIB_PATH

# status codes (thd_status_t)
OK = 0
ERR_INVALID_ARG = 1
ERR_BAD_DIRECTION = 2
ERR_CU_NONZERO_START = 3
ERR_CU_NON_MONOTONE = 4
ERR_LEN_NOT_DIVISIBLE = 5
ERR_TOTAL_MISMATCH = 6
ERR_TIMEOUT = 7
ERR_CUDA = 8
ERR_INDEX_RANGE = 9
ERR_VALID_EXCEEDS_PADDED = 10
ERR_CAPACITY = 11
ERR_SCRATCH_LIMIT = 12
PACK_NOALLOC_MAX_ROWS = 4096

STATUS_NAMES = {
    OK: "ok",
    ERR_INVALID_ARG: "invalid_arg",
    ERR_BAD_DIRECTION: "bad_direction",
    ERR_CU_NONZERO_START: "cu_nonzero_start",
    ERR_CU_NON_MONOTONE: "cu_non_monotone",
    ERR_LEN_NOT_DIVISIBLE: "len_not_divisible",
    ERR_TOTAL_MISMATCH: "total_mismatch",
    ERR_TIMEOUT: "timeout",
    ERR_CUDA: "cuda",
    ERR_INDEX_RANGE: "index_range",
    ERR_VALID_EXCEEDS_PADDED: "valid_exceeds_padded",
    ERR_CAPACITY: "capacity",
    ERR_SCRATCH_LIMIT: "scratch_limit",
}

ZIGZAG_TO_CONTIGUOUS = 0
CONTIGUOUS_TO_ZIGZAG = 1
SEQ_TO_HEAD = 0
HEAD_TO_SEQ = 1
MAX_CP = 64


class ThdRoute(ctypes.Structure):
    """Mirror of thd_route_t."""
    _fields_ = [
        ("cp_size", c_int32),
        ("dir", c_int32),
        ("total_rows", c_int64),
        ("send_rows", c_void_p),
        ("recv_rows", c_void_p),
        ("input_split_sizes", c_void_p),
        ("output_split_sizes", c_void_p),
        ("send_offsets", c_void_p),
        ("recv_offsets", c_void_p),
        ("send_identity", c_void_p),
        ("recv_identity", c_void_p),
        ("src_of_dst", c_void_p),
    ]


# name -> (restype, argtypes), one entry per function declared in include/thd.h
SIGNATURES = {
    "thd_route_bytes": (c_size_t, [c_int64, c_int32]),
    "thd_route_bind": (c_int32, [POINTER(ThdRoute), c_void_p, c_size_t, c_int64, c_int32, c_int32]),
    "thd_route_pair_bytes": (c_size_t, [c_int64, c_int32]),
    "thd_route_bind_pair": (c_int32, [POINTER(ThdRoute), POINTER(ThdRoute), c_void_p, c_size_t, c_int64, c_int32]),
    "thd_route_build": (c_int32, [c_void_p, c_int32, c_int64, c_int32, c_int32, POINTER(ThdRoute),
                                  c_void_p, c_void_p]),
    "thd_route_build_pair": (c_int32, [c_void_p, c_int32, c_int64, c_int32, POINTER(ThdRoute), POINTER(ThdRoute),
                                       c_void_p, c_void_p]),
    "thd_partition_indices": (c_int32, [c_void_p, c_int32, c_int64, c_int32, c_int32, c_void_p,
                                        c_void_p, c_void_p]),
    "thd_swap": (c_int32, [c_void_p, c_void_p, c_int64, POINTER(ThdRoute), c_void_p, c_void_p]),
    "thd_swap_batched": (c_int32, [c_void_p, c_void_p, c_int64, c_int64, POINTER(ThdRoute), c_void_p,
                                   c_void_p]),
    "thd_pack_rank": (c_int32, [c_void_p, c_void_p, c_int32, c_int64, POINTER(ThdRoute), c_void_p, c_void_p]),
    "thd_scatter_rank": (c_int32, [c_void_p, c_void_p, c_int32, c_int64, POINTER(ThdRoute), c_void_p, c_void_p]),
    "thd_pack": (c_int32, [c_void_p, c_void_p, c_int64, POINTER(ThdRoute), c_void_p, c_void_p]),
    "thd_a2a_local": (c_int32, [c_void_p, c_void_p, c_int64, POINTER(ThdRoute), c_void_p, c_void_p]),
    "thd_scatter": (c_int32, [c_void_p, c_void_p, c_int64, POINTER(ThdRoute), c_void_p, c_void_p]),
    "thd_ulysses_swap": (c_int32, [c_void_p, c_void_p, c_int64, c_int32, c_int64, c_int32, c_void_p, c_void_p]),
    "thd_roll_labels": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int64, c_int32, c_int32,
                                  c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "thd_roll_labels_zigzag": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int64, c_int32, c_int32, c_int32,
                                         c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "thd_pack_docs_workspace_bytes": (c_size_t, [c_int32, c_int64]),
    "thd_pack_docs": (c_int32, [c_void_p, c_int32, c_int64, c_int32, c_int32, c_int32, c_int32, c_int32,
                                c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_int64,
                                c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
    "thd_pack_docs_noalloc": (c_int32, [c_void_p, c_int32, c_int64, c_int32, c_int32, c_int32, c_int32, c_int32,
                                        c_void_p, c_int64, c_void_p, c_void_p, c_int64, c_void_p, c_void_p,
                                        c_void_p]),
    "thd_status_clear": (c_int32, [c_void_p, c_void_p]),
    "thd_status_read": (c_int32, [c_void_p, POINTER(c_int32), c_void_p]),
    "thd_status_string": (c_char_p, [c_int32]),
    "thd_last_cuda_error": (c_int32, []),
    "thd_version": (c_int32, []),
}

_lib = None


def load():
    """Load libthd.so (once) and declare every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{os.path.basename(path)} is not built ({path}); run `python -m context_packed_sequence_gb300.build"
            f"{' --checked' if path == CHECKED_LIB_PATH else ''}` or `__graft_entry__.build()` -- there is no CPU "
            "fallback")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
