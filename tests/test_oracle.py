"""Pins of the CPU oracle against what the pages print and what the
definitions force (runs without a GPU).

Each pin is chosen so that a plausible slip in the oracle -- the back chunk
taken as 2*cp-r, front/back swapped, a receive buffer ordered by destination
instead of source, a label reaching into padding, a trailing empty document --
fails at least one of them (the mutation tests at the end plant such slips).
"""

import itertools
import json
import os

import numpy as np
import pytest

import oracle
from oracle import thd_oracle as O
from oracle.intervals import build_route_intervals

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
Z2C, C2Z = O.ZIGZAG_TO_CONTIGUOUS, O.CONTIGUOUS_TO_ZIGZAG


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# symbol table for the worked example: ordinary tokens, EOD, raw pad, alignment pad
SYM = {c: i + 1 for i, c in enumerate("abcdefghij")}
SYM.update({"E": 99, "_": 0, "P": 77})
UNSYM = {v: k for k, v in SYM.items()}


# --------------------------------------------------------------------------
# page-printed values
# --------------------------------------------------------------------------

def test_worked_example_pack():
    g = _golden("pscp_worked_example.json")
    raw = [[SYM[s] for s in row] for row in g["raw"]]
    tokens, cu_v, cu = oracle.pack_docs(raw, eod_id=SYM["E"], align=g["align"],
                                        pad_id=SYM["P"], raw_pad_id=SYM["_"])
    assert cu_v == g["cu_seqlens"]
    assert [cu_v[i + 1] - cu_v[i] for i in range(len(cu_v) - 1)] == g["seqlens"]
    assert cu == g["cu_seqlens_padded"]
    assert [cu[i + 1] - cu[i] for i in range(len(cu) - 1)] == g["padded_seqlens"]
    assert max(cu[i + 1] - cu[i] for i in range(len(cu) - 1)) == g["max_seqlen"]
    assert [UNSYM[t] for t in tokens] == g["packed_tokens"]
    # valid_token_nums: valid tokens per raw sample (last non-pad position + 1)
    assert [sum(1 for t in row if t != SYM["_"]) for row in raw] == g["valid_token_nums"]
    _, _, valid = oracle.roll_labels(tokens, cu_v, cu, depth=0)
    assert valid == g["valid_mask"]


def test_worked_example_slice():
    g = _golden("pscp_worked_example.json")
    cu, cp = g["cu_seqlens_padded"], g["cp"]
    T = cu[-1]
    tokens = [SYM[s] for s in g["packed_tokens"]]
    valid = g["valid_mask"]
    total = 0
    for r in range(cp):
        idx = oracle.partition_indices(cu, T, cp, r)
        assert idx == g["slice_index"][r]
        assert [UNSYM[tokens[i]] for i in idx] == g["rank_tokens"][r]
        assert [valid[i] for i in idx] == g["rank_valid_mask"][r]
        assert sum(valid[i] for i in idx) == g["rank_valid_count"][r]
        total += sum(valid[i] for i in idx)
    assert total == g["total_valid"]
    # all ranks at once = the ranks' lists concatenated
    assert oracle.partition_indices(cu, T, cp, -1) == sum(g["slice_index"], [])


def test_single_document_split():
    g = _golden("pscp_single_doc_split.json")
    cu = g["cu_seqlens_padded"]
    for r in range(g["cp"]):
        assert oracle.partition_indices(cu, cu[-1], g["cp"], r) == g["slice_index"][r]


# --------------------------------------------------------------------------
# the tiny workload's route, derived by hand from the definitions
# --------------------------------------------------------------------------

def test_tiny_route_hand_derived():
    """cp=2, documents [8, 12, 4] -> cu=[0,8,20,24], S=12 rows per rank.

    Chunk sizes c = 2, 3, 1.  Rank 0 takes chunks 0 and 3 of every document:
    [0,1]+[6,7], [8,9,10]+[17,18,19], [20]+[23]; rank 1 takes chunks 1 and 2:
    [2,3]+[4,5], [11,12,13]+[14,15,16], [21]+[22].
    Contiguous rank 0 owns [0,12), rank 1 owns [12,24).
    z->c: rank 0 sends 0,1,6,7,8,9,10 to d0 (7 rows) and 17..20,23 to d1 (5);
    rank 1 sends 2,3,4,5,11 to d0 (5) and 12..16,21,22 to d1 (7).
    d0 receives from s0 then s1: slots 0,1,6,7,8,9,10 | 2,3,4,5,11.
    d1 receives 17,18,19,20,23 -> 5,6,7,8,11 | 12..16,21,22 -> 0..4,9,10.
    """
    cu, T, cp = [0, 8, 20, 24], 24, 2
    zz = O.zigzag_partition(cu, cp)
    assert zz[0] == [0, 1, 6, 7, 8, 9, 10, 17, 18, 19, 20, 23]
    assert zz[1] == [2, 3, 4, 5, 11, 12, 13, 14, 15, 16, 21, 22]
    rt = oracle.build_route(cu, T, cp, Z2C)
    ident = list(range(12))
    assert rt.send_rows == [ident, ident]
    assert rt.input_split_sizes == [[7, 5], [5, 7]]
    assert rt.output_split_sizes == [[7, 5], [5, 7]]
    assert rt.send_offsets == [[0, 7, 12], [0, 5, 12]]
    assert rt.recv_offsets == [[0, 7, 12], [0, 5, 12]]
    assert rt.recv_rows[0] == [0, 1, 6, 7, 8, 9, 10, 2, 3, 4, 5, 11]
    assert rt.recv_rows[1] == [5, 6, 7, 8, 11, 0, 1, 2, 3, 4, 9, 10]
    assert rt.send_identity == [True, True]
    assert rt.recv_identity == [False, False]
    # the fused permutation: contiguous row g comes from zigzag position of g
    zpos = {g: r * 12 + k for r in range(2) for k, g in enumerate(zz[r])}
    assert rt.src_of_dst == [zpos[g] for g in range(24)]
    # c->z is the inverse route: its send side is z->c's receive side
    back = oracle.build_route(cu, T, cp, C2Z)
    assert back.send_rows == rt.recv_rows
    assert back.recv_rows == [ident, ident]
    assert back.input_split_sizes == rt.output_split_sizes
    assert back.src_of_dst == zz[0] + zz[1]


# --------------------------------------------------------------------------
# brute force over every small packing
# --------------------------------------------------------------------------

def _compositions(cp, max_T=24, max_docs=4):
    unit = 2 * cp
    max_units = max_T // unit
    yield []
    for n in range(1, max_docs + 1):
        for parts in itertools.product(range(max_units + 1), repeat=n):
            if sum(parts) <= max_units:
                yield [unit * p for p in parts]


def _check_invariants(cu, T, cp):
    S = T // cp
    zz = O.zigzag_partition(cu, cp)
    # every rank holds T/cp rows, ascending in global order
    for r in range(cp):
        assert len(zz[r]) == S
        assert zz[r] == sorted(zz[r])
    # the zigzag layout is a partition of [0, T)
    assert sorted(sum(zz, [])) == list(range(T))
    # chunk ownership r / 2cp-1-r, and each document gives L/cp rows to each rank
    owner = {g: r for r in range(cp) for g in zz[r]}
    for i in range(len(cu) - 1):
        L = cu[i + 1] - cu[i]
        if L == 0:
            continue
        c = L // (2 * cp)
        for g in range(cu[i], cu[i + 1]):
            k = (g - cu[i]) // c
            assert owner[g] == (k if k < cp else 2 * cp - 1 - k)
        for r in range(cp):
            assert sum(1 for g in zz[r] if cu[i] <= g < cu[i + 1]) == L // cp

    routes = {}
    for direction in (Z2C, C2Z):
        rt = oracle.build_route(cu, T, cp, direction)
        routes[direction] = rt
        for s in range(cp):
            assert sum(rt.input_split_sizes[s]) == S
            assert sum(rt.output_split_sizes[s]) == S
            assert sorted(rt.send_rows[s]) == list(range(S))
            assert sorted(rt.recv_rows[s]) == list(range(S))
            for d in range(cp):
                assert rt.input_split_sizes[s][d] == rt.output_split_sizes[d][s]
        # the fused permutation is a bijection
        assert sorted(rt.src_of_dst) == list(range(T))
        # identity flags as structure dictates: z->c never reorders its send
        # side, c->z never reorders its receive side
        if direction == Z2C:
            assert all(rt.send_identity)
        else:
            assert all(rt.recv_identity)
        if cp == 1:
            assert rt.src_of_dst == list(range(T))
        assert build_route_intervals(cu, T, cp, direction) == rt

    # z->c then c->z is the identity on rows
    fwd, bwd = routes[Z2C].src_of_dst, routes[C2Z].src_of_dst
    assert [fwd[bwd[q]] for q in range(T)] == list(range(T))
    # the c->z buffer is the zigzag partition itself
    assert bwd == sum(zz, [])


def test_random_packings_keep_every_invariant():
    """Beyond the exhaustive small cases: packings of up to 24 documents
    (empty ones included) for cp = 1 .. 16, drawn by hypothesis
    (deterministically), satisfy every invariant above and agree with the
    interval-intersection reading in both directions."""
    pytest.importorskip("hypothesis")
    from hypothesis import given, settings, strategies as st

    @settings(max_examples=150, deadline=None, derandomize=True)
    @given(cp=st.integers(1, 16), units=st.lists(st.integers(0, 6), max_size=24))
    def check(cp, units):
        cu = [0]
        for u in units:
            cu.append(cu[-1] + 2 * cp * u)
        _check_invariants(cu, cu[-1], cp)

    check()


@pytest.mark.parametrize("cp", [1, 2, 3, 4])
def test_bruteforce_small_packings(cp):
    n = 0
    for lens in _compositions(cp):
        cu = [0]
        for L in lens:
            cu.append(cu[-1] + L)
        _check_invariants(cu, cu[-1], cp)
        n += 1
    assert n > 20


def test_apply_matches_fused_permutation_and_round_trips():
    rng = np.random.default_rng(7)
    for cp, lens in [(2, [8, 12, 4]), (3, [6, 0, 12, 18, 6]), (4, [16, 8, 0, 40]), (1, [2, 4])]:
        cu = [0]
        for L in lens:
            cu.append(cu[-1] + L)
        T = cu[-1]
        x = rng.integers(0, 256, size=(T, 6), dtype=np.uint8)
        rt = oracle.build_route(cu, T, cp, Z2C)
        send, recv, out = oracle.apply_route(x, rt)
        assert np.array_equal(out, x[rt.src_of_dst])
        back = oracle.build_route(cu, T, cp, C2Z)
        _, _, again = oracle.apply_route(out, back)
        assert np.array_equal(again, x)
        # contiguous rank d holds global rows [dS, (d+1)S) after z->c
        zz = O.zigzag_partition(cu, cp)
        gx = np.zeros_like(x)
        for pos, g in enumerate(sum(zz, [])):
            gx[g] = x[pos]
        assert np.array_equal(out, gx)


# --------------------------------------------------------------------------
# validation order ([PR273] 2.3, 5)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("cu,T,cp,direction,kind", [
    ([0, 8], 8, 2, 5, "bad_direction"),
    ([0, 8], 8, 0, Z2C, "invalid_arg"),
    ([0, 8], 6, 2, Z2C, "invalid_arg"),          # T not a multiple of 2cp
    ([4, 8], 8, 2, Z2C, "cu_nonzero_start"),
    ([0, 8, 4, 8], 8, 2, Z2C, "cu_non_monotone"),
    ([0, 6, 8], 8, 2, Z2C, "len_not_divisible"),
    ([0, 8], 16, 2, Z2C, "total_mismatch"),
    # precedence: start before monotone before divisible before total
    ([4, 2, 3], 8, 2, Z2C, "cu_nonzero_start"),
    ([0, 6, 4, 9], 8, 2, Z2C, "cu_non_monotone"),
    ([0, 6, 16], 8, 2, Z2C, "len_not_divisible"),
])
def test_validation_order(cu, T, cp, direction, kind):
    with pytest.raises(O.ThdValueError) as e:
        oracle.build_route(cu, T, cp, direction)
    assert e.value.kind == kind
    assert isinstance(e.value, ValueError)


def test_empty_and_degenerate_inputs():
    # T = 0 with no documents, or only empty documents, is legal
    for cu in ([0], [0, 0, 0]):
        for direction in (Z2C, C2Z):
            rt = oracle.build_route(cu, 0, 2, direction)
            assert rt.src_of_dst == [] and rt.send_rows == [[], []]
            assert rt.input_split_sizes == [[0, 0], [0, 0]]
    # repeated boundaries contribute nothing
    a = oracle.build_route([0, 8, 8, 20, 20, 24], 24, 2, Z2C)
    b = oracle.build_route([0, 8, 20, 24], 24, 2, Z2C)
    assert a == b


# --------------------------------------------------------------------------
# labels, MTP targets and the valid mask
# --------------------------------------------------------------------------

def _doc_id(cu, p):
    for i in range(len(cu) - 1):
        if cu[i] <= p < cu[i + 1]:
            return i
    raise AssertionError


def _labels_by_segment_roll(tokens, cu_v, cu, depth, fill):
    """A second reading: depth 0 is the token stream shifted left by one inside
    each padded segment with everything at or past the segment's last valid
    token blanked; depth k is depth k-1 shifted left by one inside each padded
    segment, the freed last slot blanked."""
    T = len(tokens)
    ends = []
    for i in range(len(cu) - 1):
        ends.append((cu[i], cu[i + 1], cu[i] + cu_v[i + 1] - cu_v[i]))
    lab = [fill] * T
    msk = [0] * T
    for a, b, e in ends:
        for p in range(a, b):
            if p + 1 < e:
                lab[p], msk[p] = tokens[p + 1], 1
    out_l, out_m = [lab], [msk]
    for _ in range(depth):
        prev_l, prev_m = out_l[-1], out_m[-1]
        nl, nm = [fill] * T, [0] * T
        for a, b, e in ends:
            for p in range(a, b - 1):
                nl[p], nm[p] = prev_l[p + 1], prev_m[p + 1]
        out_l.append(nl)
        out_m.append(nm)
    return out_l, out_m


def test_labels_worked_example():
    g = _golden("pscp_worked_example.json")
    raw = [[SYM[s] for s in row] for row in g["raw"]]
    tokens, cu_v, cu = oracle.pack_docs(raw, SYM["E"], g["align"], SYM["P"], SYM["_"])
    labels, lmask, valid = oracle.roll_labels(tokens, cu_v, cu, depth=0, fill=-1)
    # 13 valid tokens in 3 documents -> 10 positions have a next token
    assert sum(lmask[0]) == 13 - 3
    # the EOD positions (3, 6, 13) are masked
    for p in (3, 6, 13):
        assert tokens[p] == SYM["E"] and lmask[0][p] == 0 and labels[0][p] == -1
    # doc 0 "a b c E": labels b c E -
    assert [UNSYM.get(t, t) for t in labels[0][0:4]] == ["b", "c", "E", -1]


def test_labels_in_zigzag_layout_worked_example():
    """[PSCP] 3.6 prints each rank's valid mask after the CP slice; the labels
    sliced the same way follow from 3.8 (next token of the same document)."""
    g = _golden("pscp_worked_example.json")
    raw = [[SYM[s] for s in row] for row in g["raw"]]
    tokens, cu_v, cu = oracle.pack_docs(raw, SYM["E"], g["align"], SYM["P"], SYM["_"])
    labels, lmask, valid = oracle.roll_labels_zigzag(tokens, cu_v, cu, g["cp"], depth=1, fill=-1)
    assert valid == g["rank_valid_mask"][0] + g["rank_valid_mask"][1]
    # rank 0 holds rows 0,3,4,7,8,9,14,15 = a E d P f g P P: labels b - e - g h - -
    assert [UNSYM.get(t, t) for t in labels[0][:8]] == ["b", -1, "e", -1, "g", "h", -1, -1]
    # depth 1 for rank 1 (rows 1,2,5,6,10,11,12,13 = b c e E h i j E): d E - - j E - -
    assert [UNSYM.get(t, t) for t in labels[1][8:]] == ["E", -1, -1, -1, "j", "E", -1, -1]
    assert sum(lmask[0]) == 13 - 3
    with pytest.raises(O.ThdValueError) as e:
        oracle.roll_labels_zigzag(tokens, cu_v, [0, 4, 7, 16], 2, 0)
    assert e.value.kind == "len_not_divisible"


@pytest.mark.parametrize("depth", [0, 1, 3])
def test_labels_never_cross_documents(depth):
    rng = np.random.default_rng(11 + depth)
    for trial in range(30):
        n = int(rng.integers(0, 7))
        lv = [int(rng.integers(0, 9)) for _ in range(n)]
        lp = [L + int(rng.integers(0, 4)) for L in lv]
        cu_v, cu = [0], [0]
        for a, b in zip(lv, lp):
            cu_v.append(cu_v[-1] + a)
            cu.append(cu[-1] + b)
        T = cu[-1]
        tokens = [int(t) for t in rng.integers(0, 1000, size=T)]
        labels, lmask, valid = oracle.roll_labels(tokens, cu_v, cu, depth, fill=-5)
        assert sum(valid) == cu_v[-1]
        for k in range(depth + 1):
            for p in range(T):
                if lmask[k][p]:
                    t = p + 1 + k
                    assert _doc_id(cu, t) == _doc_id(cu, p) and valid[t] == 1
                    assert labels[k][p] == tokens[t]
                else:
                    assert labels[k][p] == -5
            # every document of valid length V has max(V-1-k, 0) targets at depth k
            assert sum(lmask[k]) == sum(max(v - 1 - k, 0) for v in lv)
        ref_l, ref_m = _labels_by_segment_roll(tokens, cu_v, cu, depth, -5)
        assert labels == ref_l and lmask == ref_m


def test_extra_token_hand_example():
    """A sample of S=6 tokens plus one extra token ([PSCP] 1.3): the document
    the sample end cuts off gets the extra token as its last label."""
    raw = [[1, 2, E, 3, 4, 5], [7, 8, 9, E, 10, E]]
    tokens, cu_v, cu, doc_next = oracle.pack_docs(raw, E, align=1, row_next=[6, 11])
    assert doc_next == [None, 6, None, None]          # row 1 ends with EOD: 11 starts a new document
    labels, lmask, _ = oracle.roll_labels(tokens, cu_v, cu, 1, fill=-1, doc_next=doc_next)
    assert labels[0] == [2, E, -1, 4, 5, 6, 8, 9, E, -1, E, -1]
    assert lmask[0] == [1, 1, 0, 1, 1, 1, 1, 1, 1, 0, 1, 0]
    assert labels[1] == [E, -1, -1, 5, 6, -1, 9, E, -1, -1, -1, -1]
    # without the extra tokens the cut document's last label is masked, as before
    assert oracle.roll_labels(tokens, cu_v, cu, 0, fill=-1)[0][0][5] == -1


def test_extra_token_matches_rolling_each_sample():
    """Second reading, as the page describes it: roll every sample left by one
    with its extra token appended, then mask the EOD positions.  Depth 0 must
    agree with the per-document definition, padded or not."""
    rng = np.random.default_rng(21)
    for trial in range(60):
        B, S = int(rng.integers(1, 5)), int(rng.integers(1, 30))
        raw = rng.integers(1, 20, size=(B, S))
        raw[rng.random((B, S)) < 0.2] = E
        raw = raw.tolist()
        extra = [int(v) for v in rng.integers(1, 20, size=B)]
        align = int(rng.choice([1, 2, 4]))
        tokens, cu_v, cu, doc_next = oracle.pack_docs(raw, E, align, pad_id=-1, row_next=extra)
        labels, lmask, valid = oracle.roll_labels(tokens, cu_v, cu, 0, fill=-9, doc_next=doc_next)
        # packed position of row b, column t: documents are laid out row by row
        got = []
        for i in range(len(cu) - 1):
            got.extend(labels[0][p] for p in range(cu[i], cu[i] + cu_v[i + 1] - cu_v[i]))
        want = []
        for b in range(B):
            rolled = raw[b][1:] + [extra[b]]
            want.extend(-9 if raw[b][t] == E else rolled[t] for t in range(S))
        assert got == want


def test_label_validation():
    with pytest.raises(O.ThdValueError) as e:
        oracle.roll_labels([1, 2, 3, 4], [0, 5], [0, 4], 0)
    assert e.value.kind == "valid_exceeds_padded"
    with pytest.raises(O.ThdValueError) as e:
        oracle.roll_labels([1, 2, 3, 4], [0, 2], [0, 8], 0)
    assert e.value.kind == "total_mismatch"


# --------------------------------------------------------------------------
# pack_docs corner cases ([PSCP] 1.11 lists them as the ones to test)
# --------------------------------------------------------------------------

E = 99


def test_pack_docs_corner_cases():
    raw = [
        [0, 0, 0, 0],          # all-pad sample: no documents
        [1, 2, E, 3],          # tail after the last EOD is a document
        [1, 2, 3, E],          # ends exactly at EOD: no empty trailing document
        [E, E, 5, 6],          # consecutive EODs: two one-token documents
        [7, 8, 9, 9],          # one document fills the whole sample, no EOD
        [4, 0, E, 0],          # pad in the middle is kept; trailing pad dropped
    ]
    tokens, cu_v, cu = oracle.pack_docs(raw, eod_id=E, align=4, pad_id=-1, raw_pad_id=0)
    lens = [cu_v[i + 1] - cu_v[i] for i in range(len(cu_v) - 1)]
    assert lens == [3, 1, 4, 1, 1, 2, 4, 3]
    assert [cu[i + 1] - cu[i] for i in range(len(cu) - 1)] == [4, 4, 4, 4, 4, 4, 4, 4]
    assert tokens[:8] == [1, 2, E, -1, 3, -1, -1, -1]
    assert tokens[-4:] == [4, 0, E, -1]


def test_pack_docs_invariants():
    rng = np.random.default_rng(3)
    for trial in range(40):
        B, S = int(rng.integers(1, 5)), int(rng.integers(1, 40))
        raw = rng.integers(1, 20, size=(B, S))
        raw[rng.random((B, S)) < 0.15] = E
        raw = raw.tolist()
        align = int(rng.choice([1, 2, 4, 16]))
        tokens, cu_v, cu = oracle.pack_docs(raw, E, align, pad_id=-1)
        assert cu_v[-1] == B * S
        stream = []
        for i in range(len(cu) - 1):
            L, P = cu_v[i + 1] - cu_v[i], cu[i + 1] - cu[i]
            assert L >= 1 and P % align == 0 and L <= P < L + align
            doc = tokens[cu[i]:cu[i] + L]
            assert all(t == -1 for t in tokens[cu[i] + L:cu[i + 1]])
            assert E not in doc[:-1]
            stream.extend(doc)
        assert stream == [t for row in raw for t in row]
        assert len(tokens) == cu[-1]


# --------------------------------------------------------------------------
# Ulysses exchange ([PSCP] 2.5, 2.7)
# --------------------------------------------------------------------------

def test_ulysses_hand_example_and_invariants():
    # 4 tokens x 2 heads of one byte, cp=2: token g is [2g, 2g+1]; rank 0 ends up
    # with every token's head 0, rank 1 with every token's head 1
    x = np.arange(8, dtype=np.uint8).reshape(4, 2)
    assert oracle.ulysses_swap(x, 2, O.SEQ_TO_HEAD).tolist() == [[0], [2], [4], [6], [1], [3], [5], [7]]
    rng = np.random.default_rng(4)
    for cp, T, H, D in [(1, 6, 3, 2), (2, 8, 4, 3), (4, 12, 8, 1), (3, 9, 6, 5)]:
        # byte (g, h, d) identifies its token and head
        x = np.zeros((T, H * D), dtype=np.uint8)
        for g in range(T):
            for h in range(H):
                x[g, h * D:(h + 1) * D] = (g * 17 + h * 5) % 251
        y = oracle.ulysses_swap(x, cp, O.SEQ_TO_HEAD)
        Hg = H // cp
        for r in range(cp):
            for g in range(T):
                # rank r holds the whole sequence, heads [r*H/cp, (r+1)*H/cp), in order
                want = [(g * 17 + h * 5) % 251 for h in range(r * Hg, (r + 1) * Hg) for _ in range(D)]
                assert y[r * T + g].tolist() == want
        assert np.array_equal(oracle.ulysses_swap(y, cp, O.HEAD_TO_SEQ), x)
        if cp == 1:
            assert np.array_equal(y, x)
        z = rng.integers(0, 256, size=(T, H * D), dtype=np.uint8)
        assert np.array_equal(oracle.ulysses_swap(oracle.ulysses_swap(z, cp, 0), cp, 1), z)
    with pytest.raises(O.ThdValueError) as e:
        oracle.ulysses_swap(x, 2, 7)
    assert e.value.kind == "bad_direction"


# --------------------------------------------------------------------------
# mutation tests: a planted slip in the oracle must fail a pin
# --------------------------------------------------------------------------

def test_mutation_back_chunk_index_is_caught(monkeypatch):
    def wrong(cu, cp):
        b = O.compact_boundaries(cu)
        zz = [[] for _ in range(cp)]
        for r in range(cp):
            for i in range(len(b) - 1):
                c = (b[i + 1] - b[i]) // (2 * cp)
                zz[r].extend(range(b[i] + r * c, b[i] + (r + 1) * c))
                back = (2 * cp - r) % (2 * cp)          # slip: 2cp-r, not 2cp-1-r
                zz[r].extend(range(b[i] + back * c, b[i] + (back + 1) * c))
        return zz
    monkeypatch.setattr(O, "zigzag_partition", wrong)
    with pytest.raises(AssertionError):
        test_worked_example_slice()


def test_mutation_receive_order_is_caught(monkeypatch):
    real = O.build_route

    def wrong(cu, T, cp, direction):
        rt = real(cu, T, cp, direction)
        # slip: receive buffer in descending source order
        S = T // cp
        for d in range(cp):
            blocks = [rt.recv_rows[d][rt.recv_offsets[d][s]:rt.recv_offsets[d][s + 1]]
                      for s in range(cp)]
            rt.recv_rows[d] = sum(reversed(blocks), [])
            rt.recv_identity[d] = rt.recv_rows[d] == list(range(S))
        return rt
    monkeypatch.setattr(O, "build_route", wrong)
    monkeypatch.setattr(oracle, "build_route", wrong)
    with pytest.raises(AssertionError):
        test_tiny_route_hand_derived()
    with pytest.raises(AssertionError):
        _check_invariants([0, 8, 20, 24], 24, 2)


def test_mutation_label_into_padding_is_caught(monkeypatch):
    def wrong(tokens, cu_v, cu, depth, fill=0):
        T = len(tokens)
        labels = [[fill] * T for _ in range(depth + 1)]
        lmask = [[0] * T for _ in range(depth + 1)]
        valid = [0] * T
        for i in range(len(cu) - 1):
            e = cu[i] + (cu_v[i + 1] - cu_v[i])
            for p in range(cu[i], cu[i + 1]):
                valid[p] = int(p < e)
                for k in range(depth + 1):
                    if p + 1 + k < cu[i + 1]:          # slip: padded end, not valid end
                        labels[k][p], lmask[k][p] = tokens[p + 1 + k], 1
        return labels, lmask, valid
    monkeypatch.setattr(oracle, "roll_labels", wrong)
    with pytest.raises(AssertionError):
        test_labels_worked_example()
