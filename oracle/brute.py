"""Pure-Python attention for tiny inputs (CPU oracle; test infrastructure only).

A triple loop over (head, query, key) with ``math`` arithmetic: the
definition of "Context parallelism and ring attention", section "The attention
problem", with the packed-THD mask of the TE tutorial sections 1 and 3 written
out pair by pair.  It shares nothing with the blocked NumPy oracle and pins it.
"""
from __future__ import annotations

import math


def attn_fwd(q, k, v, ids_q, pos_q, ids_kv, pos_kv, window_left, scale):
    """q, k: nested lists [b][s][H][d]; v: [b][s_kv][Hkv][d_v]; ids/pos [b][s].

    Returns out [b][s_q][Hq][d_v] and lse [b][Hq][s_q] as nested lists (the
    output has the width of V; d is only the width of the q.k dot product).
    """
    b, s_q, hq, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    s_kv, hkv = len(k[0]), len(k[0][0])
    dv = len(v[0][0][0])
    g = hq // hkv
    out = [[[[0.0] * dv for _ in range(hq)] for _ in range(s_q)] for _ in range(b)]
    lse = [[[-math.inf] * s_q for _ in range(hq)] for _ in range(b)]
    for bi in range(b):
        for h in range(hq):
            kh = h // g
            for i in range(s_q):
                scores = []
                for j in range(s_kv):
                    ok = (ids_q[bi][i] == ids_kv[bi][j] and ids_q[bi][i] != 0
                          and pos_kv[bi][j] <= pos_q[bi][i]
                          and (window_left < 0 or pos_q[bi][i] - pos_kv[bi][j] <= window_left))
                    if ok:
                        dot = 0.0
                        for c in range(d):
                            dot += q[bi][i][h][c] * k[bi][j][kh][c]
                        scores.append((j, scale * dot))
                if not scores:
                    continue
                big = max(sv for _, sv in scores)
                weights = [(j, math.exp(sv - big)) for j, sv in scores]
                denom = math.fsum(w for _, w in weights)
                for c in range(dv):
                    out[bi][i][h][c] = math.fsum(w * v[bi][j][kh][c] for j, w in weights) / denom
                lse[bi][h][i] = big + math.log(denom)
    return out, lse
