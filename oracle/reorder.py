"""Causal load-balancing permutations (CPU oracle; test infrastructure only).

"Context parallelism and ring attention", section "Load balance": under a
causal mask early query blocks see fewer keys than late ones, so each device
gets an early piece paired with a late piece.  Read as the dual-chunk scheme:
split the sequence into 2R equal chunks; logical shard r holds chunk r
followed by chunk 2R-1-r; shards are concatenated in order r = 0..R-1.

The TE tutorial (section 4 "Striped load balancing and sharding") uses a
striped strategy with ``stripe_size`` (1 for Ring, 512 for AllGather) but does
not define it.  Read as: cut the sequence into stripes of ``stripe_size``
tokens; stripe t goes to shard t mod R; each shard keeps its stripes in order;
shards are concatenated.

A permutation is returned as ``src``: reordered[:, i] = x[:, src[i]].
"""
from __future__ import annotations

import numpy as np

DUAL_CHUNK = 0
STRIPED = 1


def dual_chunk_src(s: int, cp_size: int) -> np.ndarray:
    if cp_size < 1 or s % (2 * cp_size):
        raise ValueError("dual-chunk reorder needs s divisible by 2*cp_size")
    c = s // (2 * cp_size)
    parts = []
    for r in range(cp_size):
        parts.append(np.arange(r * c, (r + 1) * c))
        parts.append(np.arange((2 * cp_size - 1 - r) * c, (2 * cp_size - r) * c))
    return np.concatenate(parts)


def striped_src(s: int, cp_size: int, stripe_size: int) -> np.ndarray:
    if cp_size < 1 or stripe_size < 1 or s % (cp_size * stripe_size):
        raise ValueError("striped reorder needs s divisible by cp_size*stripe_size")
    n_stripes = s // stripe_size
    parts = []
    for r in range(cp_size):
        for t in range(r, n_stripes, cp_size):
            parts.append(np.arange(t * stripe_size, (t + 1) * stripe_size))
    return np.concatenate(parts)


def src_index(s, strategy, cp_size, stripe_size=1):
    if strategy == DUAL_CHUNK:
        return dual_chunk_src(s, cp_size)
    if strategy == STRIPED:
        return striped_src(s, cp_size, stripe_size)
    raise ValueError("unknown strategy")


def reorder(x, strategy, cp_size, stripe_size=1):
    """Reorder along axis 1 (the sequence axis of [b, s, ...])."""
    x = np.asarray(x)
    return x[:, src_index(x.shape[1], strategy, cp_size, stripe_size)]


def inverse_reorder(x, strategy, cp_size, stripe_size=1):
    x = np.asarray(x)
    src = src_index(x.shape[1], strategy, cp_size, stripe_size)
    y = np.empty_like(x)
    y[:, src] = x
    return y
