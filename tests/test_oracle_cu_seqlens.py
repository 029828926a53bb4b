"""Pins for the oracle's segment_ids -> cu_seqlens conversion (no GPU).

The conversion is RFC-0025 "支持 Attention Varlen 功能并对齐 Loss", 方案 §1.
Pins: the page's four worked examples; the cumulative-length definition of
"Drill: Sequence Packing from scratch" (数学 / The math) applied to the
generator's own document lengths; an exhaustive brute-force check of the
properties that define cu_seqlens (doc(s) = i iff cu[i] <= s < cu[i+1]) on
every id array of length <= 7 over {0,1,2,3}; and the two amendments, which
must agree with the page's reading wherever the page's reading is sound.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
import synth


def _read_examples(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            seg, ms, cu = (p.strip() for p in line.split(";"))
            rows.append(([int(x) for x in seg.split(",")], int(ms), [int(x) for x in cu.split(",")]))
    return rows


def test_worked_examples(golden_dir):
    rows = _read_examples(os.path.join(golden_dir, "cu_seqlens_examples.txt"))
    assert len(rows) == 4
    for seg, ms, expected in rows:
        for frs, er in [(True, "last_real"), (False, "count")]:
            cu, n = oracle.cu_seqlens(np.array([seg], np.int32), ms, force_row_starts=frs,
                                      end_rule=er)
            assert cu.tolist() == expected, (seg, frs, er)


def _lengths_to_cu(lengths, max_segs):
    # Drill definition: cu[0] = 0, cu[i] = sum_{j<=i} l_j; phantoms repeat the total
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    while len(cu) < max_segs + 1:
        cu.append(cu[-1])
    return cu


@pytest.mark.parametrize("name", ["tiny", "b2", "ling3", "short", "long"])
def test_matches_cumulative_length_definition(name):
    wl = synth.WORKLOADS[name]
    seg, lengths = synth.make_segment_ids(wl, synth.default_seed(name))
    flat_lengths = [L for row in lengths for L in row]
    assert sum(flat_lengths) == int((seg != 0).sum())
    cu, n = oracle.cu_seqlens(seg, wl.max_segs)
    assert n == len(flat_lengths)
    assert n <= wl.max_segs
    assert cu.tolist() == _lengths_to_cu(flat_lengths, wl.max_segs)
    if name == "tiny":
        assert cu.tolist() == [0, 100, 137, 256, 256]


def _check_defining_properties(seg_flat, T, max_segs, cu, n_segs):
    """Properties that pin cu_seqlens down when n_segs <= max_segs."""
    N = len(seg_flat)
    assert cu[0] == 0
    assert all(cu[i] <= cu[i + 1] for i in range(max_segs))
    real = [p for p in range(N) if seg_flat[p] != 0]
    n_end = (real[-1] + 1) if real else 0
    # segment rank of each real token: number of starts at or before it, minus one
    rank = []
    r = -1
    for p in range(N):
        if seg_flat[p] != 0 and (p % T == 0 or seg_flat[p] != seg_flat[p - 1]):
            r += 1
        rank.append(r)
    assert n_segs == r + 1
    if n_segs <= max_segs:
        for p in real:
            i = rank[p]
            assert cu[i] <= p < cu[i + 1], (seg_flat, p, cu)
        # the last real segment ends one past the last real token; phantoms are empty
        for i in range(max(n_segs, 1), max_segs + 1):
            assert cu[i] == n_end
        # interior segment ends coincide with the next segment's first token
        for i in range(1, n_segs):
            p = cu[i]
            assert seg_flat[p] != 0 and rank[p] == i and (p % T == 0 or seg_flat[p] != seg_flat[p - 1])
    else:
        # overflow: the first max_segs-1 ends are exact, the last slot ends at N
        assert cu[max_segs] == N
        for i in range(1, max_segs):
            p = cu[i]
            assert rank[p] == i and (p % T == 0 or seg_flat[p] != seg_flat[p - 1])


def test_bruteforce_small_arrays():
    count = 0
    for L in range(1, 8):
        for seg in itertools.product(range(4), repeat=L):
            arr = np.array([seg], np.int32)
            for ms in (1, 2, 3, 5):
                cu, n = oracle.cu_seqlens(arr, ms)
                _check_defining_properties(list(seg), L, ms, cu.tolist(), n)
                count += 1
    assert count > 20000


def test_bruteforce_two_rows():
    rng = np.random.default_rng(7)
    for _ in range(3000):
        T = int(rng.integers(1, 7))
        seg = rng.integers(0, 3, size=(2, T)).astype(np.int32)
        ms = int(rng.integers(1, 6))
        cu, n = oracle.cu_seqlens(seg, ms)
        _check_defining_properties(seg.reshape(-1).tolist(), T, ms, cu.tolist(), n)


def test_amendments_agree_with_page_reading_when_sound():
    """With one row and padding only at the tail, the page's flat scan and
    its count of real tokens give the same cu_seqlens as the amended rules."""
    rng = np.random.default_rng(3)
    for _ in range(500):
        T = int(rng.integers(1, 40))
        seg = synth.random_segment_ids(rng, 1, T, max_len=6)
        pad = int(rng.integers(0, 4))
        if pad:
            seg[0, T - min(pad, T):] = 0
        ms = int(rng.integers(1, 12))
        a = oracle.cu_seqlens(seg, ms, force_row_starts=True, end_rule="last_real")
        b = oracle.cu_seqlens(seg, ms, force_row_starts=False, end_rule="count")
        assert a[0].tolist() == b[0].tolist() and a[1] == b[1]


def test_amendment_a_row_start_collision():
    # two rows whose documents share id 1: the page's flat scan merges them,
    # the forced row start keeps them apart (RFC-0026 §3.1.1: t = 0 always starts)
    seg = np.array([[1, 1, 1], [1, 1, 1]], np.int32)
    cu_a, n_a = oracle.cu_seqlens(seg, 4, force_row_starts=True)
    cu_p, n_p = oracle.cu_seqlens(seg, 4, force_row_starts=False)
    assert n_a == 2 and cu_a.tolist() == [0, 3, 6, 6, 6]
    assert n_p == 1 and cu_p.tolist() == [0, 6, 6, 6, 6]


def test_amendment_b_interior_padding():
    # padding at the end of row 0: counting real tokens would end the last
    # segment at 5 and cut off token 5 of the second row's document
    seg = np.array([[1, 1, 0], [1, 1, 1]], np.int32)
    cu_a, _ = oracle.cu_seqlens(seg, 3)
    cu_c, _ = oracle.cu_seqlens(seg, 3, end_rule="count")
    assert cu_a.tolist() == [0, 3, 6, 6]
    assert cu_c.tolist() == [0, 3, 5, 5]


def test_overflow_merges_into_last_slot():
    seg = np.array([[1, 2, 3, 4, 5, 0]], np.int32)
    cu, n = oracle.cu_seqlens(seg, 3)
    assert n == 5
    assert cu.tolist() == [0, 1, 2, 6]


def test_all_padding_and_empty():
    cu, n = oracle.cu_seqlens(np.zeros((2, 5), np.int32), 3)
    assert n == 0 and cu.tolist() == [0, 0, 0, 0]
    cu, n = oracle.cu_seqlens(np.zeros((1, 0), np.int32), 2)
    assert n == 0 and cu.tolist() == [0, 0, 0]
