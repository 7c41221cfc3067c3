"""Exact packed-THD attention in float64 (CPU oracle; test infrastructure only).

Definition followed ("Context parallelism and ring attention", section "The
attention problem"): for one head, O = softmax(Q K^T / sqrt(H) + M) V, where M
is 0 on visible pairs and -inf elsewhere.  H is the head dimension, as the TE
tutorial's ``scaling_factor=head_dim**-0.5`` (section 3 "Fused attention
call") fixes; the scale is passed in explicitly.

The mask M for a PADDING_CAUSAL mask with a (left, 0) sliding window over a
segment-id / segment-pos descriptor (TE tutorial, section 1 "Packed THD
inputs" and section 3) is read as:

    visible(i, j)  <=>  ids_q[i] == ids_kv[j] != 0
                        and pos_kv[j] <= pos_q[i]
                        and (W < 0 or pos_q[i] - pos_kv[j] <= W)

id 0 marks padding; positions, not array indices, decide causality and the
window (the window is inclusive: W + 1 keys including the query itself).

The softmax is taken in one shot over all visible keys of a row (no online
rescaling).  Rows with no visible key get O = 0 and LSE = -inf.  LSE is the
natural log of the softmax denominator including the scale:
LSE_i = ln sum_j exp(scale * q_i . k_j) over visible j.

GQA: query head h reads kv head h // (Hq // Hkv).

Layouts: q/out/dout [b, s_q, Hq, d]; k/v [b, s_kv, Hkv, d]; ids/pos [b, s];
lse [b, Hq, s_q].  Inputs may be torch tensors (any dtype) or numpy arrays;
they are converted exactly to float64.
"""
from __future__ import annotations

import numpy as np

ROW_BLOCK = 256


def _f64(x):
    if hasattr(x, "detach"):
        import torch
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x):
    if hasattr(x, "detach"):
        return x.detach().cpu().numpy().astype(np.int64)
    return np.asarray(x).astype(np.int64)


def visible(ids_q, pos_q, ids_kv, pos_kv, window_left):
    """Boolean mask [len(ids_q), len(ids_kv)] of visible (query, key) pairs."""
    iq = np.asarray(ids_q, dtype=np.int64)[:, None]
    pq = np.asarray(pos_q, dtype=np.int64)[:, None]
    ik = np.asarray(ids_kv, dtype=np.int64)[None, :]
    pk = np.asarray(pos_kv, dtype=np.int64)[None, :]
    m = (iq == ik) & (iq != 0) & (pk <= pq)
    if window_left >= 0:
        m &= (pq - pk) <= window_left
    return m


def count_pairs(ids_q, pos_q, ids_kv, pos_kv, window_left):
    """Exact number of visible (query, key) pairs of one batch row.

    Counted per query row: the keys of the same nonzero segment whose position
    lies in [pos_q - W, pos_q] (or <= pos_q without a window).
    """
    iq, pq = _i64(ids_q), _i64(pos_q)
    ik, pk = _i64(ids_kv), _i64(pos_kv)
    total = 0
    for sid in np.unique(iq):
        if sid == 0:
            continue
        keys = np.sort(pk[ik == sid])
        if keys.size == 0:
            continue
        qp = pq[iq == sid]
        hi = np.searchsorted(keys, qp, side="right")
        if window_left >= 0:
            lo = np.searchsorted(keys, qp - window_left, side="left")
        else:
            lo = np.zeros_like(hi)
        total += int(np.sum(hi - lo))
    return total


def _row_blocks(rows, block=ROW_BLOCK):
    rows = np.asarray(rows, dtype=np.int64)
    for i in range(0, rows.size, block):
        yield rows[i:i + block]


def attn_fwd(q, k, v, ids_q, pos_q, ids_kv, pos_kv, window_left, scale,
             *, batches=None, heads=None, rows=None):
    """Forward attention.  Returns (out, lse) in float64.

    ``batches``/``heads``/``rows`` restrict the computation to a subset of
    batch rows, query heads and query rows (the other entries stay 0 / -inf);
    each computed row is exact regardless of the subset.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    ids_q, pos_q, ids_kv, pos_kv = map(_i64, (ids_q, pos_q, ids_kv, pos_kv))
    b, s_q, hq, d = q.shape
    hkv = k.shape[2]
    dv = v.shape[3]  # O takes V's width; d is the q.k contraction width only
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    g = hq // hkv
    out = np.zeros((b, s_q, hq, dv))
    lse = np.full((b, hq, s_q), -np.inf)
    batches = range(b) if batches is None else batches
    heads = range(hq) if heads is None else heads
    rows = np.arange(s_q) if rows is None else np.asarray(rows)
    for bi in batches:
        for blk in _row_blocks(rows):
            mask = visible(ids_q[bi, blk], pos_q[bi, blk], ids_kv[bi], pos_kv[bi], window_left)
            cols = np.nonzero(mask.any(axis=0))[0]
            if cols.size == 0:
                continue
            m = mask[:, cols]
            has = m.any(axis=1)
            for h in heads:
                kvh = h // g
                s = scale * (q[bi, blk, h, :] @ k[bi, cols, kvh, :].T)
                s = np.where(m, s, -np.inf)
                mx = np.where(has, s.max(axis=1), 0.0)
                e = np.where(m, np.exp(s - mx[:, None]), 0.0)
                z = e.sum(axis=1)
                zsafe = np.where(has, z, 1.0)
                p = e / zsafe[:, None]
                out[bi, blk, h, :] = p @ v[bi, cols, kvh, :]
                lse[bi, h, blk] = np.where(has, mx + np.log(zsafe), -np.inf)
    return out, lse


def attn_bwd(q, k, v, dout, ids_q, pos_q, ids_kv, pos_kv, window_left, scale,
             *, out=None, batches=None, kv_heads=None, rows=None):
    """Gradient of loss = sum(out * dout) with respect to q, k, v (float64).

    Uses the explicit probability matrix P of each row:
        dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),
        dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q,
    with dK / dV summed over the query heads that share a kv head.  The TE
    tutorial (section 5 "Ring and AllGather") differentiates exactly this loss
    (a vdot of the output with dout), so dout is the output gradient.

    ``out``: the forward output used for D (defaults to the exact float64
    output).  ``rows`` restricts the query rows that contribute: dQ is exact on
    those rows; dK/dV hold only the contributions of those rows (complete for
    any key whose visible queries all lie in ``rows``).  ``kv_heads`` restricts
    the groups computed.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    ids_q, pos_q, ids_kv, pos_kv = map(_i64, (ids_q, pos_q, ids_kv, pos_kv))
    b, s_q, hq, d = q.shape
    hkv = k.shape[2]
    g = hq // hkv
    if out is None:
        heads = None if kv_heads is None else [h for kh in kv_heads for h in range(kh * g, kh * g + g)]
        out, _ = attn_fwd(q, k, v, ids_q, pos_q, ids_kv, pos_kv, window_left, scale,
                          batches=batches, heads=heads, rows=rows)
    else:
        out = _f64(out)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    batches = range(b) if batches is None else batches
    kv_heads = range(hkv) if kv_heads is None else kv_heads
    rows = np.arange(s_q) if rows is None else np.asarray(rows)
    for bi in batches:
        for blk in _row_blocks(rows):
            mask = visible(ids_q[bi, blk], pos_q[bi, blk], ids_kv[bi], pos_kv[bi], window_left)
            cols = np.nonzero(mask.any(axis=0))[0]
            if cols.size == 0:
                continue
            m = mask[:, cols]
            has = m.any(axis=1)
            for kvh in kv_heads:
                kk = k[bi, cols, kvh, :]
                vv = v[bi, cols, kvh, :]
                for h in range(kvh * g, kvh * g + g):
                    s = scale * (q[bi, blk, h, :] @ kk.T)
                    s = np.where(m, s, -np.inf)
                    mx = np.where(has, s.max(axis=1), 0.0)
                    e = np.where(m, np.exp(s - mx[:, None]), 0.0)
                    z = np.where(has, e.sum(axis=1), 1.0)
                    p = e / z[:, None]
                    do = dout[bi, blk, h, :]
                    dv[bi, cols, kvh, :] += p.T @ do
                    dp = do @ vv.T
                    dd = np.sum(do * out[bi, blk, h, :], axis=1)
                    ds = p * (dp - dd[:, None])
                    dq[bi, blk, h, :] = scale * (ds @ kk)
                    dk[bi, cols, kvh, :] += scale * (ds.T @ q[bi, blk, h, :])
    return dq, dk, dv


def rows_seeing_keys(ids_q, pos_q, ids_kv, pos_kv, window_left, key_rows):
    """Query rows (one batch row) that see at least one of ``key_rows``."""
    m = visible(_i64(ids_q), _i64(pos_q), _i64(ids_kv)[key_rows], _i64(pos_kv)[key_rows],
                window_left)
    return np.nonzero(m.any(axis=1))[0]
