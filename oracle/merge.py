"""Running-softmax merge (CPU oracle; test infrastructure only).

"Context parallelism and ring attention", section "Online softmax": each query
row keeps m (largest score seen), z (sum of exponentials relative to m) and u
(exponential-weighted value sum).  A new block (m_b, z_b, u_b) is folded in by

    m' = max(m, m_b)
    z' = e^(m - m') z + e^(m_b - m') z_b
    u' = e^(m - m') u + e^(m_b - m') u_b

and after all blocks the output is u' / z'.  A block with no visible key has
m = -inf, z = 0, u = 0 and contributes nothing.

A finished partial result (O, LSE) of attention over some key block is the
triple (m = LSE, z = 1, u = O): u / z = O and m + ln z = LSE.  ``merge_partial``
folds two such results with the update above and returns (O', LSE') with
LSE' = m' + ln z'.
"""
from __future__ import annotations

import numpy as np


def _scale(m, m_new):
    """e^(m - m_new), defined as 0 when m = -inf (no keys seen yet)."""
    out = np.zeros(np.broadcast(m, m_new).shape)
    ok = np.isfinite(m) & np.isfinite(m_new)
    np.exp(np.where(ok, m - np.where(ok, m_new, 0.0), 0.0), out=out, where=ok)
    return out


def merge_mzu(m, z, u, m_b, z_b, u_b):
    """One online-softmax update.  m, z: [...]; u: [..., d].  Returns (m', z', u')."""
    m, z, u = np.asarray(m, float), np.asarray(z, float), np.asarray(u, float)
    m_b, z_b, u_b = np.asarray(m_b, float), np.asarray(z_b, float), np.asarray(u_b, float)
    m_new = np.maximum(m, m_b)
    a = _scale(m, m_new)
    c = _scale(m_b, m_new)
    return m_new, a * z + c * z_b, a[..., None] * u + c[..., None] * u_b


def block_stats(scores, visible_mask, values):
    """(m_b, z_b, u_b) of one key block for a set of query rows.

    scores [r, n] (already scaled), visible_mask [r, n], values [n, d].
    """
    s = np.where(visible_mask, scores, -np.inf)
    has = visible_mask.any(axis=1)
    m_b = np.where(has, s.max(axis=1, initial=-np.inf), -np.inf)
    e = np.where(visible_mask, np.exp(s - np.where(has, m_b, 0.0)[:, None]), 0.0)
    return m_b, e.sum(axis=1), e @ values


def finish(m, z, u):
    """Output u / z and LSE m + ln z; (0, -inf) for rows that saw no key."""
    has = z > 0
    zs = np.where(has, z, 1.0)
    out = np.where(has[..., None], u / zs[..., None], 0.0)
    lse = np.where(has, m + np.log(zs), -np.inf)
    return out, lse


def merge_partial(out_acc, lse_acc, out_blk, lse_blk):
    """Merge two finished partial results given as (O, LSE).

    out_*: [b, s, H, d]; lse_*: [b, H, s] (the library's layouts).
    Returns (O', LSE') in float64.
    """
    oa = np.asarray(out_acc, float)
    ob = np.asarray(out_blk, float)
    la = np.transpose(np.asarray(lse_acc, float), (0, 2, 1))   # [b, s, H]
    lb = np.transpose(np.asarray(lse_blk, float), (0, 2, 1))
    za = np.where(np.isfinite(la), 1.0, 0.0)
    zb = np.where(np.isfinite(lb), 1.0, 0.0)
    ua = np.where(np.isfinite(la)[..., None], oa, 0.0)
    ub = np.where(np.isfinite(lb)[..., None], ob, 0.0)
    m, z, u = merge_mzu(la, za, ua, lb, zb, ub)
    out, lse = finish(m, z, u)
    return out, np.transpose(lse, (0, 2, 1))
