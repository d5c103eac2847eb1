"""CPU oracle of the THD context-parallel layout conversion.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg, never by the product package, which
fails loudly when its CUDA library is missing instead of falling back here.
"""

from .thd_oracle import (  # noqa: F401
    ZIGZAG_TO_CONTIGUOUS, CONTIGUOUS_TO_ZIGZAG, ThdValueError, Route,
    validate_route_args, compact_boundaries, zigzag_partition, contiguous_partition,
    partition_indices, build_route, pack, all_to_all, scatter, apply_route,
    validate_label_args, roll_labels, roll_labels_zigzag, pack_docs,
    SEQ_TO_HEAD, HEAD_TO_SEQ, ulysses_swap,
)
