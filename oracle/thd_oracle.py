"""Per-token CPU oracle of the packed-sequence (THD) context-parallel layout conversion.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the CUDA library computes.  Only the test-suite, the smoke
check and the benchmark's CPU-baseline leg may import it; the product path
never does, and this module imports nothing from the product package.

Pure Python integers and lists throughout.  NumPy appears only as byte storage
for payload rows (``apply_route``), never for index arithmetic.  Every value
here is an integer or a raw byte, so the result is exact: the GPU must match it
bit for bit.

Sources (web pages, cited by title and section):

* [PR273] "[Task32] feat: fla mcore chunkwise cp stage 3" (Relax PR #273),
  section 2.1 (the route: both layouts are unions of global token intervals,
  contiguous = one interval per rank, zigzag = 2 x num_docs intervals per
  rank; pack with ``send_rows``, all-to-all with the split sizes, scatter with
  ``recv_rows``), section 2.2 (identity rows mean zero-copy; repeated
  boundaries are empty padding slots and are dropped), section 2.3 and
  section 5 (fail-fast ``ValueError`` on a length not divisible by 2*cp, on
  ``cu_seqlens`` not starting at 0, on a non-monotone ``cu_seqlens`` and on an
  invalid direction).
* [PSCP] "Packed Sequence 与上下文并行" (Packed sequences and context
  parallelism), section 1.3 (labels roll without crossing a sample),
  section 1.6 (MTP rolls must not cross a document), section 2.2 (pack: split
  at EOD, pad every document to the alignment, flatten), section 2.4 (ring
  zigzag split: each document cut into 2*cp chunks, rank r owns chunk r and
  chunk 2*cp-1-r), section 3 (the worked example B=2, S=8, CP=2) and
  section 3.8 (the EOD position's label is masked).

Readings taken where the pages are silent:

* contiguous layout: rank r holds the global rows [r*T/cp, (r+1)*T/cp)
  ([PR273] 2.1 "one interval per rank"; [PSCP] 2.5 slices Ulysses the same way);
* inside one (source, destination) block rows keep ascending global order;
  the send buffer is grouped by destination in ascending rank order and the
  receive buffer by source in ascending rank order (all-to-all concatenation);
* the route is driven by the padded ``cu_seqlens``; every padded length must be
  a multiple of 2*cp;
* the label of position p at MTP depth k (k = 0 is the ordinary label) is
  ``tokens[p+1+k]`` when p+1+k is still a valid (non-pad) position of the same
  document, else ``fill`` with loss-mask 0.
"""

from __future__ import annotations

from dataclasses import dataclass, field

ZIGZAG_TO_CONTIGUOUS = 0
CONTIGUOUS_TO_ZIGZAG = 1

# Failure kinds, named after the checks of [PR273] 2.3 / 5 plus argument checks.
BAD_DIRECTION = "bad_direction"
INVALID_ARG = "invalid_arg"
CU_NONZERO_START = "cu_nonzero_start"
CU_NON_MONOTONE = "cu_non_monotone"
LEN_NOT_DIVISIBLE = "len_not_divisible"
TOTAL_MISMATCH = "total_mismatch"
VALID_EXCEEDS_PADDED = "valid_exceeds_padded"


class ThdValueError(ValueError):
    """A fail-fast validation error; ``kind`` names the failed check."""

    def __init__(self, kind: str, message: str):
        super().__init__(message)
        self.kind = kind


# --------------------------------------------------------------------------
# validation ([PR273] 2.3 and 5)
# --------------------------------------------------------------------------

def validate_route_args(cu, T, cp, direction):
    """Raise ThdValueError for the first failed check, in this order:

    direction; cp >= 1; T >= 0 and T a multiple of 2*cp (T is the row count of
    the packed tensor, known without reading cu); cu non-empty; cu[0] == 0;
    cu non-decreasing (lowest offending index first); every document length a
    multiple of 2*cp (lowest document first); cu[-1] == T.
    """
    if direction not in (ZIGZAG_TO_CONTIGUOUS, CONTIGUOUS_TO_ZIGZAG):
        raise ThdValueError(BAD_DIRECTION, f"invalid THD layout direction {direction!r}")
    if cp < 1:
        raise ThdValueError(INVALID_ARG, f"cp_size must be >= 1, got {cp}")
    if T < 0 or T % (2 * cp) != 0:
        raise ThdValueError(INVALID_ARG, f"T={T} is not a non-negative multiple of 2*cp={2 * cp}")
    if len(cu) < 1:
        raise ThdValueError(INVALID_ARG, "cu_seqlens must hold at least one boundary")
    if cu[0] != 0:
        raise ThdValueError(CU_NONZERO_START, f"cu_seqlens must start at 0, got {cu[0]}")
    for i in range(len(cu) - 1):
        if cu[i + 1] < cu[i]:
            raise ThdValueError(CU_NON_MONOTONE, f"cu_seqlens is not monotone at index {i + 1}")
    for i in range(len(cu) - 1):
        if (cu[i + 1] - cu[i]) % (2 * cp) != 0:
            raise ThdValueError(
                LEN_NOT_DIVISIBLE,
                f"sequence {i} has length {cu[i + 1] - cu[i]}, not divisible by 2*cp={2 * cp} "
                "for zigzag/contiguous THD partitioning")
    if cu[-1] != T:
        raise ThdValueError(TOTAL_MISMATCH, f"cu_seqlens[-1]={cu[-1]} does not equal T={T}")


def compact_boundaries(cu):
    """Drop repeated boundaries: an empty document is an empty padding slot
    that owns no rows ([PR273] 2.2)."""
    out = [cu[0]]
    for b in cu[1:]:
        if b != out[-1]:
            out.append(b)
    return out


# --------------------------------------------------------------------------
# layouts ([PSCP] 2.4, [PR273] 2.1)
# --------------------------------------------------------------------------

def zigzag_partition(cu, cp):
    """zz[r] = the global rows rank r holds in the zigzag layout, in local order.

    Each document of padded length L is cut into 2*cp chunks of c = L/(2*cp)
    rows; rank r takes chunk r (front) then chunk 2*cp-1-r (back), documents in
    order ([PSCP] 2.4).
    """
    b = compact_boundaries(cu)
    zz = [[] for _ in range(cp)]
    for r in range(cp):
        for i in range(len(b) - 1):
            c = (b[i + 1] - b[i]) // (2 * cp)
            front = b[i] + r * c
            back = b[i] + (2 * cp - 1 - r) * c
            zz[r].extend(range(front, front + c))
            zz[r].extend(range(back, back + c))
    return zz


def contiguous_partition(T, cp):
    """cont[r] = [r*T/cp, (r+1)*T/cp): one interval per rank ([PR273] 2.1)."""
    S = T // cp
    return [list(range(r * S, (r + 1) * S)) for r in range(cp)]


def partition_indices(cu, T, cp, rank=-1):
    """Global row held in each local slot of the zigzag layout.

    rank >= 0: the list for that rank (what the pages' ``get_slice_index`` /
    ``thd_get_partitioned_indices`` return).  rank == -1: all ranks
    concatenated rank-major, i.e. the global zigzag buffer's source rows.
    """
    validate_route_args(cu, T, cp, ZIGZAG_TO_CONTIGUOUS)
    zz = zigzag_partition(cu, cp)
    if rank == -1:
        out = []
        for r in range(cp):
            out.extend(zz[r])
        return out
    if not 0 <= rank < cp:
        raise ThdValueError(INVALID_ARG, f"cp_rank {rank} out of range for cp_size {cp}")
    return list(zz[rank])


# --------------------------------------------------------------------------
# route ([PR273] 2.1, 2.2, 2.4): built token by token
# --------------------------------------------------------------------------

@dataclass
class Route:
    cp: int
    T: int
    direction: int
    send_rows: list = field(default_factory=list)           # [cp][S]
    recv_rows: list = field(default_factory=list)           # [cp][S]
    input_split_sizes: list = field(default_factory=list)   # [s][d] rows s sends to d
    output_split_sizes: list = field(default_factory=list)  # [d][s] rows d receives from s
    send_offsets: list = field(default_factory=list)        # [s][cp+1]
    recv_offsets: list = field(default_factory=list)        # [d][cp+1]
    send_identity: list = field(default_factory=list)       # [cp] bool
    recv_identity: list = field(default_factory=list)       # [cp] bool
    src_of_dst: list = field(default_factory=list)          # [T]


def _exclusive_prefix(row):
    out = [0]
    for v in row:
        out.append(out[-1] + v)
    return out


def build_route(cu, T, cp, direction):
    """The all-to-all route that turns layout A into layout B.

    z->c: A = zigzag, B = contiguous; c->z: A = contiguous, B = zigzag.
    Every source row k of rank s holds global token g = A[s][k]; it goes to the
    rank d that owns g in layout B, into slot ownerB(g).  Rows are bucketed by
    destination, scanning source slots in order, so each bucket keeps the
    source's order (ascending global order, since both layouts list every
    rank's rows ascending).  The receive side takes the buckets of source 0,
    1, ... in turn.
    """
    validate_route_args(cu, T, cp, direction)
    S = T // cp
    zz = zigzag_partition(cu, cp)
    cont = contiguous_partition(T, cp)
    if direction == ZIGZAG_TO_CONTIGUOUS:
        A, B = zz, cont
    else:
        A, B = cont, zz

    owner_b = {}
    for r in range(cp):
        for k, g in enumerate(B[r]):
            owner_b[g] = (r, k)

    bucket = [[[] for _ in range(cp)] for _ in range(cp)]
    for s in range(cp):
        for k, g in enumerate(A[s]):
            d = owner_b[g][0]
            bucket[s][d].append(k)

    rt = Route(cp=cp, T=T, direction=direction)
    for s in range(cp):
        rows = []
        for d in range(cp):
            rows.extend(bucket[s][d])
        rt.send_rows.append(rows)
        rt.input_split_sizes.append([len(bucket[s][d]) for d in range(cp)])
    for d in range(cp):
        rt.output_split_sizes.append([rt.input_split_sizes[s][d] for s in range(cp)])
        rows = []
        for s in range(cp):
            for k in bucket[s][d]:
                rows.append(owner_b[A[s][k]][1])
        rt.recv_rows.append(rows)
    rt.send_offsets = [_exclusive_prefix(r) for r in rt.input_split_sizes]
    rt.recv_offsets = [_exclusive_prefix(r) for r in rt.output_split_sizes]
    rt.send_identity = [rt.send_rows[r] == list(range(S)) for r in range(cp)]
    rt.recv_identity = [rt.recv_rows[r] == list(range(S)) for r in range(cp)]

    # The fused permutation over the two global buffers: target position
    # d*S + slot receives source position s*S + k.
    src = [-1] * T
    for s in range(cp):
        for k, g in enumerate(A[s]):
            d, slot = owner_b[g]
            src[d * S + slot] = s * S + k
    rt.src_of_dst = src
    return rt


# --------------------------------------------------------------------------
# applying a route, every virtual rank simulated in turn ([PR273] 2.1)
# --------------------------------------------------------------------------

def pack(x, route):
    """send[s][j] = x[s][send_rows[s][j]]; x is a [cp*S, row_bytes] uint8 array."""
    cp, S = route.cp, route.T // route.cp
    send = x.copy()
    for s in range(cp):
        for j in range(S):
            send[s * S + j] = x[s * S + route.send_rows[s][j]]
    return send


def all_to_all(send, route):
    """recv[d][recv_off[d][s] + m] = send[s][send_off[s][d] + m], m < n[s][d]."""
    cp, S = route.cp, route.T // route.cp
    recv = send.copy()
    for d in range(cp):
        for s in range(cp):
            n = route.input_split_sizes[s][d]
            for m in range(n):
                recv[d * S + route.recv_offsets[d][s] + m] = send[s * S + route.send_offsets[s][d] + m]
    return recv


def scatter(recv, route):
    """out[d][recv_rows[d][j]] = recv[d][j]."""
    cp, S = route.cp, route.T // route.cp
    out = recv.copy()
    for d in range(cp):
        for j in range(S):
            out[d * S + route.recv_rows[d][j]] = recv[d * S + j]
    return out


def apply_route(x, route):
    """pack -> all-to-all -> scatter; returns (send, recv, out)."""
    send = pack(x, route)
    recv = all_to_all(send, route)
    out = scatter(recv, route)
    return send, recv, out


# --------------------------------------------------------------------------
# Ulysses: sequence shards <-> head shards ([PSCP] 2.5, 2.7)
# --------------------------------------------------------------------------

SEQ_TO_HEAD = 0
HEAD_TO_SEQ = 1


def ulysses_swap(x, cp, direction):
    """x: [T, row_bytes] uint8 (SEQ_TO_HEAD) or [cp*T, row_bytes/cp] (HEAD_TO_SEQ).

    Ulysses slices the packed sequence into cp contiguous shards ([PSCP] 2.5)
    and its all-to-all leaves every rank the whole sequence for a subset of
    the heads ([PSCP] 2.7).  Reading: rank r gets head group r, the r-th of cp
    equal slices of each token row.  One piece at a time:
    SEQ_TO_HEAD: out[r*T + g] = x[g][r*P:(r+1)*P];  HEAD_TO_SEQ: the inverse.
    """
    import numpy as np  # byte storage only

    if direction not in (SEQ_TO_HEAD, HEAD_TO_SEQ):
        raise ThdValueError(BAD_DIRECTION, f"invalid Ulysses direction {direction!r}")
    if cp < 1:
        raise ThdValueError(INVALID_ARG, f"cp_size must be >= 1, got {cp}")
    if direction == SEQ_TO_HEAD:
        T, row = x.shape
        if T % cp or row % cp:
            raise ThdValueError(INVALID_ARG, "T and the row must split into cp parts")
        P = row // cp
        out = np.zeros((cp * T, P), dtype=x.dtype)
        for r in range(cp):
            for g in range(T):
                out[r * T + g] = x[g, r * P:(r + 1) * P]
        return out
    rows, P = x.shape
    if rows % cp or (rows // cp) % cp:
        raise ThdValueError(INVALID_ARG, "rows must split into cp ranks of a multiple of cp tokens")
    T = rows // cp
    out = np.zeros((T, cp * P), dtype=x.dtype)
    for r in range(cp):
        for g in range(T):
            out[g, r * P:(r + 1) * P] = x[r * T + g]
    return out


# --------------------------------------------------------------------------
# labels, MTP targets and the valid mask ([PSCP] 1.3, 1.6, 3.8)
# --------------------------------------------------------------------------

def _check_cu_plain(cu, T, name):
    if len(cu) < 1:
        raise ThdValueError(INVALID_ARG, f"{name} must hold at least one boundary")
    if cu[0] != 0:
        raise ThdValueError(CU_NONZERO_START, f"{name} must start at 0, got {cu[0]}")
    for i in range(len(cu) - 1):
        if cu[i + 1] < cu[i]:
            raise ThdValueError(CU_NON_MONOTONE, f"{name} is not monotone at index {i + 1}")
    if T is not None and cu[-1] != T:
        raise ThdValueError(TOTAL_MISMATCH, f"{name}[-1]={cu[-1]} does not equal T={T}")


def validate_label_args(cu_v, cu, T, depth):
    """Checks, in order: depth >= 0; T >= 0; both boundary lists the same
    length; padded boundaries (start 0, monotone, total T); unpadded
    boundaries (start 0, monotone); every valid length <= its padded length."""
    if depth < 0 or T < 0:
        raise ThdValueError(INVALID_ARG, "mtp depth and T must be >= 0")
    if len(cu_v) != len(cu):
        raise ThdValueError(INVALID_ARG, "cu_seqlens and cu_seqlens_padded differ in length")
    _check_cu_plain(cu, T, "cu_seqlens_padded")
    _check_cu_plain(cu_v, None, "cu_seqlens")
    for i in range(len(cu) - 1):
        if cu_v[i + 1] - cu_v[i] > cu[i + 1] - cu[i]:
            raise ThdValueError(VALID_EXCEEDS_PADDED,
                                f"sequence {i}: valid length exceeds padded length")


def roll_labels(tokens, cu_v, cu, depth, fill=0, doc_next=None):
    """labels[k][p], loss_mask[k][p] for k = 0..depth, and valid[p].

    Position p of document i (cu[i] <= p < cu[i+1]) is valid when
    p < e_i = cu[i] + (cu_v[i+1] - cu_v[i]), i.e. it is a real token and not
    alignment padding ([PSCP] 2.2, valid_local_token_mask).  Its depth-k
    target is tokens[p+1+k] when p+1+k < e_i: the target never reaches past
    the document's last valid token into padding or into the next document
    ([PSCP] 1.3, 1.6).  Otherwise the label is ``fill`` and the mask 0 -- in
    particular at the EOD position itself ([PSCP] 3.8).

    doc_next (optional, one entry per document, None or a token id): a
    document cut by the end of its sample continues with the sample's extra
    token ([PSCP] 1.3, ``last_extra_token``).  Its token stream is then the
    valid tokens followed by that one token, so the target p+1+k == e_i is
    doc_next[i] (mask 1) and only targets beyond it are ``fill``.
    """
    T = len(tokens)
    validate_label_args(cu_v, cu, T, depth)
    if doc_next is not None and len(doc_next) != len(cu) - 1:
        raise ThdValueError(INVALID_ARG, "doc_next needs one entry per document")
    labels = [[fill] * T for _ in range(depth + 1)]
    lmask = [[0] * T for _ in range(depth + 1)]
    valid = [0] * T
    for i in range(len(cu) - 1):
        e = cu[i] + (cu_v[i + 1] - cu_v[i])
        nxt = None if doc_next is None else doc_next[i]
        for p in range(cu[i], cu[i + 1]):
            valid[p] = 1 if p < e else 0
            for k in range(depth + 1):
                t = p + 1 + k
                if t < e:
                    labels[k][p] = tokens[t]
                    lmask[k][p] = 1
                elif t == e and nxt is not None:
                    labels[k][p] = nxt
                    lmask[k][p] = 1
    return labels, lmask, valid


def roll_labels_zigzag(tokens, cu_v, cu, cp, depth, fill=0, doc_next=None):
    """roll_labels, then the zigzag slicing of every output ([PSCP] 2.4 slices
    tokens, labels, loss mask and valid mask with the same index): position
    r*S + j holds the values of global row partition_indices(cu, T, cp, r)[j].

    Checks: the route's checks for (cu, T, cp) first, then the label checks."""
    T = len(tokens)
    validate_route_args(cu, T, cp, ZIGZAG_TO_CONTIGUOUS)
    labels, lmask, valid = roll_labels(tokens, cu_v, cu, depth, fill, doc_next)
    idx = partition_indices(cu, T, cp, -1)
    return ([[row[g] for g in idx] for row in labels],
            [[row[g] for g in idx] for row in lmask],
            [valid[g] for g in idx])


# --------------------------------------------------------------------------
# pack raw rows into one padded THD sequence ([PSCP] 2.2, 3.2-3.4)
# --------------------------------------------------------------------------

def pack_docs(raw, eod_id, align, pad_id=0, raw_pad_id=None, row_next=None):
    """Split each raw row into documents and flatten them with alignment padding.

    raw: list of B rows of token ids.  A row's valid region ends after its last
    token that is not ``raw_pad_id`` (the whole row when raw_pad_id is None).
    Inside it, every EOD closes a document and belongs to it; a non-empty tail
    after the last EOD is a document as well; documents never span rows.  Each
    document of length L is padded with ``pad_id`` to L + ((-L) mod align).

    Returns (tokens, cu_seqlens, cu_seqlens_padded); with ``row_next`` (one
    extra token per row, the sample's ``last_extra_token`` of [PSCP] 1.3)
    also doc_next: per document, the extra token of its row when the document
    is that row's last one, reaches the row's end (no trailing pad) and does
    not end with EOD, else None.
    """
    if align < 1:
        raise ThdValueError(INVALID_ARG, f"align must be >= 1, got {align}")
    docs = []
    doc_next = []
    for b, row in enumerate(raw):
        ve = len(row)
        if raw_pad_id is not None:
            ve = 0
            for t in range(len(row)):
                if row[t] != raw_pad_id:
                    ve = t + 1
        cur = []
        for t in range(ve):
            cur.append(row[t])
            if row[t] == eod_id:
                docs.append(cur)
                doc_next.append(None)
                cur = []
        if cur:
            docs.append(cur)
            continued = row_next is not None and ve == len(row)
            doc_next.append(row_next[b] if continued else None)
    cu_v = [0]
    cu = [0]
    tokens = []
    for d in docs:
        L = len(d)
        P = L + ((-L) % align)
        cu_v.append(cu_v[-1] + L)
        cu.append(cu[-1] + P)
        tokens.extend(d)
        tokens.extend([pad_id] * (P - L))
    if row_next is not None:
        return tokens, cu_v, cu, doc_next
    return tokens, cu_v, cu
