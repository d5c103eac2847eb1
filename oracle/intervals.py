"""Second, independent reading of the route: interval intersection.

TEST INFRASTRUCTURE ONLY (imported by the tests, never by the product path).

"[Task32] feat: fla mcore chunkwise cp stage 3" (Relax PR #273), section 2.1,
describes the route without any per-token index: both layouts are unions of
global token intervals (contiguous: one per rank; zigzag: two per document per
rank), so the rows that rank s sends to rank d are the intersection of s's
source intervals with d's target intervals, found by walking the two sorted
interval lists with two pointers, then expanded into row numbers.

``thd_oracle.build_route`` builds the same route token by token with an owner
map.  The two share no code; the tests require them to agree exactly, which
pins the ordering conventions (ascending global order inside a block,
destination-major send buffer, source-major receive buffer).
"""

from __future__ import annotations

from .thd_oracle import Route, ZIGZAG_TO_CONTIGUOUS, validate_route_args


def zigzag_segments(cu, cp, r):
    """Rank r's zigzag intervals [start, end), in local order, empty ones skipped."""
    segs = []
    for i in range(len(cu) - 1):
        L = cu[i + 1] - cu[i]
        if L == 0:
            continue
        c = L // (2 * cp)
        segs.append((cu[i] + r * c, cu[i] + (r + 1) * c))
        segs.append((cu[i] + (2 * cp - 1 - r) * c, cu[i] + (2 * cp - r) * c))
    return segs


def contiguous_segments(T, cp, r):
    S = T // cp
    return [(r * S, (r + 1) * S)] if S > 0 else []


def intersect(a_segs, b_segs):
    """Two-pointer intersection of two ascending, disjoint interval lists."""
    out = []
    i = j = 0
    while i < len(a_segs) and j < len(b_segs):
        lo = max(a_segs[i][0], b_segs[j][0])
        hi = min(a_segs[i][1], b_segs[j][1])
        if lo < hi:
            out.append((lo, hi))
        if a_segs[i][1] <= b_segs[j][1]:
            i += 1
        else:
            j += 1
    return out


def local_slots(segs, start, end):
    """Local slots of the global rows [start, end) inside a rank's interval list."""
    base = 0
    for s0, s1 in segs:
        if s0 <= start and end <= s1:
            return list(range(base + start - s0, base + end - s0))
        base += s1 - s0
    raise AssertionError("interval not inside the rank's segments")


def build_route_intervals(cu, T, cp, direction):
    validate_route_args(cu, T, cp, direction)
    S = T // cp
    zz = [zigzag_segments(cu, cp, r) for r in range(cp)]
    ct = [contiguous_segments(T, cp, r) for r in range(cp)]
    A, B = (zz, ct) if direction == ZIGZAG_TO_CONTIGUOUS else (ct, zz)
    # A layout lists every rank's intervals in local order; both layouts have
    # them ascending, which the two-pointer walk needs.
    blocks = [[intersect(A[s], B[d]) for d in range(cp)] for s in range(cp)]
    rt = Route(cp=cp, T=T, direction=direction)
    for s in range(cp):
        rows = []
        sizes = []
        for d in range(cp):
            n = 0
            for lo, hi in blocks[s][d]:
                rows.extend(local_slots(A[s], lo, hi))
                n += hi - lo
            sizes.append(n)
        rt.send_rows.append(rows)
        rt.input_split_sizes.append(sizes)
    for d in range(cp):
        rows = []
        for s in range(cp):
            for lo, hi in blocks[s][d]:
                rows.extend(local_slots(B[d], lo, hi))
        rt.recv_rows.append(rows)
        rt.output_split_sizes.append([rt.input_split_sizes[s][d] for s in range(cp)])
    for table, dest in ((rt.input_split_sizes, rt.send_offsets),
                        (rt.output_split_sizes, rt.recv_offsets)):
        for row in table:
            acc = [0]
            for v in row:
                acc.append(acc[-1] + v)
            dest.append(acc)
    rt.send_identity = [rt.send_rows[r] == list(range(S)) for r in range(cp)]
    rt.recv_identity = [rt.recv_rows[r] == list(range(S)) for r in range(cp)]
    src = [-1] * T
    for s in range(cp):
        for d in range(cp):
            for lo, hi in blocks[s][d]:
                ks = local_slots(A[s], lo, hi)
                qs = local_slots(B[d], lo, hi)
                for k, q in zip(ks, qs):
                    src[d * S + q] = s * S + k
    rt.src_of_dst = src
    return rt
