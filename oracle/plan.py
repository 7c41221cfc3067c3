"""Per-tile work classification (CPU oracle; test infrastructure only).

"Context parallelism and ring attention", section "Causal attention": a block
of keys entirely in the future of a block of queries is skipped, a block that
is entirely valid is processed without a mask, and overlapping ranges get an
element mask.  Generalised to packed segments, padding and a left window, per
(batch row, 128-query tile, 128-key tile):

  SKIP     no pair can be visible, decided from per-tile summaries: either
           tile holds only padding; the nonzero id ranges do not intersect;
           every key position lies after every query position
           (min pos_kv > max pos_q); or every key is further back than the
           window (max pos_kv < min pos_q - W).
  FULL     every pair is visible: both tiles are complete, hold no padding and
           one common nonzero id, max pos_kv <= min pos_q, and (W < 0 or
           max pos_q - min pos_kv <= W).
  PARTIAL  otherwise (needs the element mask).

Summaries (per tile): whether any token is valid (id != 0); whether any slot
is padding or lies past the end of the sequence; min / max nonzero id; min /
max position over valid tokens.

The rule is conservative: it never skips a tile that holds a visible pair and
never marks FULL a tile that holds an invisible one; ``brute_classes``
computes the exact classification from the element mask for comparison.
"""
from __future__ import annotations

import numpy as np

from .attention import visible

TILE = 128
SKIP, PARTIAL, FULL = 0, 1, 2


def summaries(ids, pos, tile=TILE):
    """Per-tile summaries of one batch row: dict of arrays over tiles."""
    ids = np.asarray(ids, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    s = ids.size
    n = -(-s // tile)
    out = {k: np.zeros(n, dtype=np.int64) for k in
           ("any_valid", "has_pad", "id_min", "id_max", "pos_min", "pos_max")}
    for t in range(n):
        sl = slice(t * tile, min((t + 1) * tile, s))
        ti, tp = ids[sl], pos[sl]
        valid = ti != 0
        out["has_pad"][t] = int((~valid).any() or ti.size < tile)
        if valid.any():
            out["any_valid"][t] = 1
            out["id_min"][t] = ti[valid].min()
            out["id_max"][t] = ti[valid].max()
            out["pos_min"][t] = tp[valid].min()
            out["pos_max"][t] = tp[valid].max()
    return out


def classes(ids_q, pos_q, ids_kv, pos_kv, window_left, tile=TILE):
    """Rule-based class array [b, n_q_tiles, n_kv_tiles] (uint8)."""
    ids_q, pos_q = np.asarray(ids_q), np.asarray(pos_q)
    ids_kv, pos_kv = np.asarray(ids_kv), np.asarray(pos_kv)
    b = ids_q.shape[0]
    nq = -(-ids_q.shape[1] // tile)
    nk = -(-ids_kv.shape[1] // tile)
    cls = np.zeros((b, nq, nk), dtype=np.uint8)
    for bi in range(b):
        sq = summaries(ids_q[bi], pos_q[bi], tile)
        sk = summaries(ids_kv[bi], pos_kv[bi], tile)
        for a in range(nq):
            skip = (
                (sq["any_valid"][a] == 0) | (sk["any_valid"] == 0)
                | (sq["id_max"][a] < sk["id_min"]) | (sk["id_max"] < sq["id_min"][a])
                | (sk["pos_min"] > sq["pos_max"][a])
            )
            if window_left >= 0:
                skip |= sk["pos_max"] < sq["pos_min"][a] - window_left
            full = (
                (sq["has_pad"][a] == 0) & (sk["has_pad"] == 0)
                & (sq["id_min"][a] == sq["id_max"][a])
                & (sk["id_min"] == sk["id_max"]) & (sk["id_min"] == sq["id_min"][a])
                & (sk["pos_max"] <= sq["pos_min"][a])
            )
            if window_left >= 0:
                full &= (sq["pos_max"][a] - sk["pos_min"]) <= window_left
            row = np.full(nk, PARTIAL, dtype=np.uint8)
            row[full] = FULL
            row[skip] = SKIP
            cls[bi, a] = row
    return cls


def ranges(cls):
    """Per (b, q tile): [first, last] kv tile that is not SKIP; (0, -1) if none."""
    b, nq, nk = cls.shape
    rng = np.zeros((b, nq, 2), dtype=np.int64)
    for bi in range(b):
        for a in range(nq):
            nz = np.nonzero(cls[bi, a] != SKIP)[0]
            rng[bi, a] = (nz[0], nz[-1]) if nz.size else (0, -1)
    return rng


def brute_classes(ids_q, pos_q, ids_kv, pos_kv, window_left, tile=TILE):
    """Exact classification from the element mask (small inputs only)."""
    ids_q, pos_q = np.asarray(ids_q), np.asarray(pos_q)
    ids_kv, pos_kv = np.asarray(ids_kv), np.asarray(pos_kv)
    b, s_q = ids_q.shape
    s_kv = ids_kv.shape[1]
    nq, nk = -(-s_q // tile), -(-s_kv // tile)
    cls = np.zeros((b, nq, nk), dtype=np.uint8)
    for bi in range(b):
        m = visible(ids_q[bi], pos_q[bi], ids_kv[bi], pos_kv[bi], window_left)
        for a in range(nq):
            for c in range(nk):
                blk = m[a * tile:(a + 1) * tile, c * tile:(c + 1) * tile]
                if not blk.any():
                    cls[bi, a, c] = SKIP
                elif blk.all() and blk.shape == (tile, tile):
                    cls[bi, a, c] = FULL
                else:
                    cls[bi, a, c] = PARTIAL
    return cls
