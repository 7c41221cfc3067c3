"""Pins for the length -> segment descriptor oracle (CPU)."""
import numpy as np
import pytest

import workload
from oracle.descriptors import segments_from_seqlens


def test_tutorial_slots_equal_the_workload_descriptor():
    """TE tutorial section 1: 4 slots of 16384 with 12288 valid tokens each is
    lengths [12288]*4 at offsets 0, 16384, 32768, 49152 — the same ids/pos as
    the tutorial's own construction (workload.segments)."""
    ids, pos = segments_from_seqlens([[12288] * 4] * 2, 65536,
                                     offsets=[[0, 16384, 32768, 49152]] * 2)
    wi, wp = workload.segments(2, 65536, 4)
    np.testing.assert_array_equal(ids, wi.numpy())
    np.testing.assert_array_equal(pos, wp.numpy())


def test_bshd_rows_one_segment_each():
    ids, pos = segments_from_seqlens([[5], [0], [8]], 8)
    np.testing.assert_array_equal(ids, [[1] * 5 + [0] * 3, [0] * 8, [1] * 8])
    np.testing.assert_array_equal(pos, [list(range(8))] * 3)


def test_packed_varlen_by_hand():
    """Back-to-back segments (cumulative-length form), an empty one and a
    tail of padding, written out by hand."""
    ids, pos = segments_from_seqlens([[3, 0, 5]], 10)
    np.testing.assert_array_equal(ids[0], [1, 1, 1, 3, 3, 3, 3, 3, 0, 0])
    np.testing.assert_array_equal(pos[0], [0, 1, 2, 0, 1, 2, 3, 4, 5, 6])


def test_gaps_before_and_between_segments_by_hand():
    ids, pos = segments_from_seqlens([[2, 3]], 9, offsets=[[2, 6]])
    np.testing.assert_array_equal(ids[0], [0, 0, 1, 1, 0, 0, 2, 2, 2])
    np.testing.assert_array_equal(pos[0], [0, 1, 0, 1, 2, 3, 0, 1, 2])


def test_truncated_at_row_end_and_negative_lengths():
    ids, pos = segments_from_seqlens([[4, -3, 10]], 8)
    np.testing.assert_array_equal(ids[0], [1, 1, 1, 1, 3, 3, 3, 3])
    np.testing.assert_array_equal(pos[0], [0, 1, 2, 3, 0, 1, 2, 3])


@pytest.mark.parametrize("seed", range(5))
def test_matches_brute_force_loop(seed):
    """Against a direct per-token walk over the segments."""
    rng = np.random.default_rng(seed)
    b, nseg, s = 3, 7, 97
    lens = rng.integers(-2, 25, size=(b, nseg))
    gaps = rng.integers(0, 6, size=(b, nseg))
    offs = np.cumsum(gaps + np.maximum(lens, 0), axis=1) - np.maximum(lens, 0)
    for offsets in (None, offs):
        ids, pos = segments_from_seqlens(lens, s, offsets)
        for bi in range(b):
            start = 0
            starts = []
            for j in range(nseg):
                starts.append(start if offsets is None else int(offsets[bi, j]))
                start += max(int(lens[bi, j]), 0)
            for t in range(s):
                cand = [j for j in range(nseg) if starts[j] <= t]
                if not cand:
                    assert (ids[bi, t], pos[bi, t]) == (0, t)
                    continue
                j = cand[-1]
                rel = t - starts[j]
                want = j + 1 if rel < max(int(lens[bi, j]), 0) else 0
                assert (ids[bi, t], pos[bi, t]) == (want, rel), (bi, t)
