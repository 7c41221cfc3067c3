"""Segment descriptors from sequence lengths (CPU oracle; test infrastructure only).

TE tutorial, section 1 "Packed THD inputs": a SequenceDescriptor built from
segment ids and positions tells the attention which tokens of a packed row
belong to which segment (ids 1, 2, ...; positions counted from each segment's
first token) and which slots are padding (id 0).  The TE Cpp attention page
("I/O Contract") takes per-row sequence lengths instead (seqlen_q,
seqlen_kv), and BSHD batches are rows with one segment each.  This module
turns lengths, with optional start offsets, into the id/pos form:

* row bi holds segments j = 0..nseg-1; segment j starts at offsets[bi, j]
  (non-decreasing) or, without offsets, right after the previous one
  (offsets = exclusive running sum of the lengths), and covers
  max(seqlens[bi, j], 0) tokens;
* token t belongs to the last segment j with offsets[bi, j] <= t; it gets
  pos = t - offsets[bi, j] and id = j + 1 if pos < that segment's length,
  else id 0 (padding after the segment, pos still counted from its start);
  a token before every segment start is padding with pos = t.

The tutorial's packed row (4 slots of 16384 tokens, 12288 valid) is
seqlens = [12288] * 4 with offsets = [0, 16384, 32768, 49152]: ids 1..4 on
valid tokens, 0 on padding, pos = index inside the slot.
"""
from __future__ import annotations

import numpy as np


def segments_from_seqlens(seqlens, s: int, offsets=None):
    """ids, pos as int32 [b, s] for lengths [b, nseg] (and offsets [b, nseg])."""
    lens = np.maximum(np.asarray(seqlens, dtype=np.int64), 0)
    if lens.ndim != 2 or lens.shape[1] < 1:
        raise ValueError("seqlens must be [b, nseg] with nseg >= 1")
    b, nseg = lens.shape
    if offsets is None:
        starts = np.concatenate([np.zeros((b, 1), np.int64), np.cumsum(lens, axis=1)[:, :-1]],
                                axis=1)
    else:
        starts = np.asarray(offsets, dtype=np.int64)
        if starts.shape != lens.shape:
            raise ValueError("offsets must have the shape of seqlens")
    ids = np.zeros((b, s), np.int32)
    pos = np.zeros((b, s), np.int32)
    t = np.arange(s, dtype=np.int64)
    for bi in range(b):
        # last segment index whose start is <= t (starts are non-decreasing)
        j = np.searchsorted(starts[bi], t, side="right") - 1
        before = j < 0
        jj = np.where(before, 0, j)
        rel = t - starts[bi][jj]
        inside = ~before & (rel < lens[bi][jj])
        ids[bi] = np.where(inside, jj + 1, 0)
        pos[bi] = np.where(before, t, rel)
    return ids, pos
