"""Packed-sequence (THD) context-parallel layout conversion for one GB300.

All cp virtual context-parallel ranks live in one device buffer, so the
zigzag <-> contiguous all-to-all is an on-device row permutation.  The CUDA
library ``libthd.so`` (C ABI in ``include/thd.h``) does all the work; this
package is its thin torch binding.
"""

from .api import (  # noqa: F401
    ZIGZAG_TO_CONTIGUOUS, CONTIGUOUS_TO_ZIGZAG, SEQ_TO_HEAD, HEAD_TO_SEQ, ThdError, Route, RouteCache,
    new_status, status_clear, status_read, check_status,
    route_build, route_build_pair, partition_indices, swap, swap_seq_dim, pack, a2a_local, scatter,
    pack_rank, scatter_rank, ulysses_swap,
    roll_labels, roll_labels_zigzag, pack_docs, zigzag_contiguous_thd_swap,
)
from .exchange import CpExchange  # noqa: F401
from . import _lib  # noqa: F401

__version__ = "0.1.0"
