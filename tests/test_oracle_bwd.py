"""Pins for the backward oracle (CPU only): finite differences and the
invariants that follow from softmax rows summing to one."""
import numpy as np
import pytest
import torch

import workload
from oracle import attention as A


def _loss(q, k, v, dout, ids, pos, w, scale):
    out, _ = A.attn_fwd(q, k, v, ids, pos, ids, pos, w, scale)
    return float(np.sum(out * dout))


@pytest.mark.parametrize("window,random_pack", [(-1, False), (3, True)])
def test_bwd_central_finite_differences(window, random_pack):
    b, s, hq, hkv, d = 1, 12, 4, 2, 3
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=17, with_dout=True)
    if random_pack:
        ids, pos = workload.random_segments(b, s, seed=4, max_segments=3, pad_prob=0.2)
    else:
        ids, pos = workload.segments(b, s, None)
    qn, kn, vn, don = (x.to(torch.float64).numpy() for x in (q, k, v, dout))
    ids, pos = ids.numpy(), pos.numpy()
    scale = 0.7
    dq, dk, dv = A.attn_bwd(qn, kn, vn, don, ids, pos, ids, pos, window, scale)
    eps = 1e-6
    for name, x, g in (("q", qn, dq), ("k", kn, dk), ("v", vn, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": qn, "k": kn, "v": vn}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], don, ids, pos, window, scale)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], don, ids, pos, window, scale)
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g, num, atol=2e-7, err_msg=name)


def test_bwd_invariants():
    b, s, hq, hkv, d = 2, 96, 6, 2, 8
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=23, with_dout=True)
    ids, pos = workload.random_segments(b, s, seed=23)
    dq, dk, dv = A.attn_bwd(q, k, v, dout, ids, pos, ids, pos, 10, 0.4)
    out, lse = A.attn_fwd(q, k, v, ids, pos, ids, pos, 10, 0.4)
    do = dout.to(torch.float64).numpy()
    g = hq // hkv
    for bi in range(b):
        valid = np.isfinite(lse[bi, 0])  # rows with >= 1 visible key
        for kh in range(hkv):
            # sum_j dV_j = sum over rows with a visible key of dO_i (P rows sum to 1)
            want = sum(do[bi, valid, h, :].sum(0) for h in range(kh * g, kh * g + g))
            np.testing.assert_allclose(dv[bi, :, kh].sum(0), want, atol=1e-10)
            # sum_j dK_j = 0 within each segment (softmax shift invariance)
            for sid in np.unique(ids[bi].numpy()):
                if sid == 0:
                    continue
                sel = (ids[bi] == sid).numpy()
                np.testing.assert_allclose(dk[bi, sel, kh].sum(0), 0.0, atol=1e-10)
        pad = (ids[bi] == 0).numpy()
        assert np.all(dq[bi, pad] == 0) and np.all(dk[bi, pad] == 0) and np.all(dv[bi, pad] == 0)


def test_bwd_row_subset_is_exact_for_dq_and_for_covered_keys():
    b, s, hq, hkv, d = 1, 200, 4, 1, 8
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=29, with_dout=True)
    ids, pos = workload.segments(b, s, 2)
    full = A.attn_bwd(q, k, v, dout, ids, pos, ids, pos, 30, 0.3)
    keys = np.arange(40, 48)
    rows = A.rows_seeing_keys(ids[0], pos[0], ids[0], pos[0], 30, keys)
    part = A.attn_bwd(q, k, v, dout, ids, pos, ids, pos, 30, 0.3, rows=rows)
    np.testing.assert_allclose(part[0][0, rows], full[0][0, rows], atol=1e-12)
    np.testing.assert_allclose(part[1][0, keys], full[1][0, keys], atol=1e-12)
    np.testing.assert_allclose(part[2][0, keys], full[2][0, keys], atol=1e-12)
