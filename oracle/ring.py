"""Ring attention over R logical shards (CPU oracle; test infrastructure only).

"Context parallelism and ring attention", section "Ring attention": each
shard keeps its query block; at every step it attends to the key/value block
currently held, folds the result into a running softmax (section "Online
softmax") and passes the block on, until every block has been seen.  Here the
R shards live in one process: shard r at step t holds block j = (r - t) mod R
(its own block first).  The sequence is first put in causal load-balancing
order (section "Load balance"), and the result is put back in natural order.
Masks use the segment positions, which travel with the tokens, so causality
across shard boundaries is decided by global position.
"""
from __future__ import annotations

import numpy as np

from . import reorder as ro
from .attention import _f64, _i64, visible
from .merge import block_stats, finish, merge_mzu


def ring_attention(q, k, v, ids, pos, window_left, scale, cp_size,
                   strategy=ro.DUAL_CHUNK, stripe_size=1):
    """Returns (out [b,s,Hq,d], lse [b,Hq,s]) in natural token order."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    ids, pos = _i64(ids), _i64(pos)
    b, s, hq, d = q.shape
    hkv = k.shape[2]
    g = hq // hkv
    qr, kr, vr = (ro.reorder(x, strategy, cp_size, stripe_size) for x in (q, k, v))
    ir, pr = (ro.reorder(x, strategy, cp_size, stripe_size) for x in (ids, pos))
    n = s // cp_size
    out = np.zeros_like(qr)
    lse = np.full((b, hq, s), -np.inf)
    for bi in range(b):
        for r in range(cp_size):
            rq = slice(r * n, (r + 1) * n)
            m = np.full((hq, n), -np.inf)
            z = np.zeros((hq, n))
            u = np.zeros((hq, n, d))
            for t in range(cp_size):
                j = (r - t) % cp_size
                rk = slice(j * n, (j + 1) * n)
                mask = visible(ir[bi, rq], pr[bi, rq], ir[bi, rk], pr[bi, rk], window_left)
                for h in range(hq):
                    kvh = h // g
                    sc = scale * (qr[bi, rq, h, :] @ kr[bi, rk, kvh, :].T)
                    mb, zb, ub = block_stats(sc, mask, vr[bi, rk, kvh, :])
                    m[h], z[h], u[h] = merge_mzu(m[h], z[h], u[h], mb, zb, ub)
            o, l = finish(m, z, u)
            out[bi, rq] = np.transpose(o, (1, 0, 2))
            lse[bi, :, rq] = l
    out = ro.inverse_reorder(out, strategy, cp_size, stripe_size)
    lse = np.transpose(ro.inverse_reorder(np.transpose(lse, (0, 2, 1)), strategy,
                                          cp_size, stripe_size), (0, 2, 1))
    return out, lse
