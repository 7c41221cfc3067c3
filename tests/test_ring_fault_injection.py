"""Host-side fault injection for the ring schedule (CPU, oracle pieces only).

A ring step that drops, duplicates or repeats a key/value block must be
caught: the merged result then differs from full attention, and the number of
(query, key) pairs each shard folded in differs from the exact visible-pair
count of its rows ("Context parallelism and ring attention", section "Ring
attention": every local query must see every allowed block exactly once)."""
import numpy as np
import pytest

import workload
from oracle import attention as A
from oracle import merge as M
from oracle import reorder as RO


def _ring(q, k, v, ids, pos, R, schedule, window=-1, scale=0.3):
    """Ring over R shards with a given block schedule per shard.
    Returns (out, lse, pairs_folded_per_shard)."""
    q, k, v = (x.double().numpy() for x in (q, k, v))
    ids, pos = ids.numpy(), pos.numpy()
    s = q.shape[1]
    src = RO.dual_chunk_src(s, R)
    qr, kr, vr, ir, pr = q[:, src], k[:, src], v[:, src], ids[:, src], pos[:, src]
    n = s // R
    out = np.zeros_like(qr)
    folded = []
    for r in range(R):
        rq = slice(r * n, (r + 1) * n)
        m = np.full(n, -np.inf)
        z = np.zeros(n)
        u = np.zeros((n, q.shape[3]))
        pairs = 0
        for j in schedule(r):
            rk = slice(j * n, (j + 1) * n)
            vis = A.visible(ir[0, rq], pr[0, rq], ir[0, rk], pr[0, rk], window)
            sc = scale * (qr[0, rq, 0] @ kr[0, rk, 0].T)
            mb, zb, ub = M.block_stats(sc, vis, vr[0, rk, 0])
            m, z, u = M.merge_mzu(m, z, u, mb, zb, ub)
            pairs += int(vis.sum())
        o, _ = M.finish(m, z, u)
        out[0, rq, 0] = o
        expected = A.count_pairs(ir[0, rq], pr[0, rq], ir[0], pr[0], window)
        folded.append((pairs, expected))
    return RO.inverse_reorder(out, RO.DUAL_CHUNK, R), folded


@pytest.mark.parametrize("fault", ["none", "drop", "duplicate", "repeat_local"])
def test_ring_fault_is_detected(fault):
    R, s = 4, 64
    q, k, v = workload.qkv(1, s, 1, 1, 8, seed=41)
    ids, pos = workload.segments(1, s, None)

    def schedule(r):
        order = [(r - t) % R for t in range(R)]
        if fault == "drop" and r == 2:
            order = order[:-1]                 # a block never arrives
        if fault == "duplicate" and r == 3:
            order = order + [order[1]]         # a block is folded in twice
        if fault == "repeat_local" and r == 1:
            order = [r] * R                    # the ring never rotates
        return order

    out, folded = _ring(q, k, v, ids, pos, R, schedule)
    full, _ = A.attn_fwd(q, k, v, ids, pos, ids, pos, -1, 0.3)
    tally_ok = all(p == e for p, e in folded)
    result_ok = np.allclose(out, full, atol=1e-12)
    if fault == "none":
        assert tally_ok and result_ok
    else:
        assert not tally_ok          # the pair tally flags the faulty shard
        assert not result_ok         # and the output is indeed wrong
