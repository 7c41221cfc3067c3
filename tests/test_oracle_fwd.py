"""Pins for the forward oracle (CPU only).

Each test checks the oracle against something other than itself: the
pure-Python brute force, closed forms, invariants, or a library routine.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workload
from oracle import attention as A
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _nested(x):
    return x.to(torch.float64).tolist()


def _small(seed, b=1, s=40, hq=4, hkv=2, d=8, slots=None, random_pack=False, dv=None):
    q, k, v = workload.qkv(b, s, hq, hkv, d, seed=seed, dv=dv)
    if random_pack:
        ids, pos = workload.random_segments(b, s, seed=seed)
    else:
        ids, pos = workload.segments(b, s, slots)
    return q, k, v, ids, pos


@pytest.mark.parametrize("seed,window,random_pack,slots", [
    (1, -1, False, None), (2, 5, False, None), (3, -1, True, None),
    (4, 3, True, None), (5, 0, True, None), (6, -1, False, 4), (7, 7, False, 2),
])
def test_blocked_matches_brute_force(seed, window, random_pack, slots):
    q, k, v, ids, pos = _small(seed, random_pack=random_pack, slots=slots)
    scale = 8 ** -0.5
    out, lse = A.attn_fwd(q, k, v, ids, pos, ids, pos, window, scale)
    bo, bl = brute.attn_fwd(_nested(q), _nested(k), _nested(v), ids.tolist(), pos.tolist(),
                            ids.tolist(), pos.tolist(), window, scale)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    bl = np.array(bl)
    assert np.array_equal(np.isinf(lse), np.isinf(bl))
    fin = np.isfinite(bl)
    np.testing.assert_allclose(lse[fin], bl[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("d,dv,window", [(12, 8, -1), (6, 10, 4)])
def test_value_width_differs_from_qk_width(d, dv, window):
    """O takes V's head dim (MLA-style d_qk != d_v): brute force and the
    library SDPA, which both take V's width as given."""
    q, k, v, ids, pos = _small(21 + d, b=2, s=36, d=d, dv=dv, random_pack=True)
    scale = d ** -0.5
    out, lse = A.attn_fwd(q, k, v, ids, pos, ids, pos, window, scale)
    assert out.shape == (2, 36, 4, dv)
    bo, bl = brute.attn_fwd(_nested(q), _nested(k), _nested(v), ids.tolist(), pos.tolist(),
                            ids.tolist(), pos.tolist(), window, scale)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    for bi in range(2):
        mask = torch.from_numpy(A.visible(ids[bi].numpy(), pos[bi].numpy(),
                                          ids[bi].numpy(), pos[bi].numpy(), window))
        qq = q[bi].to(torch.float64).permute(1, 0, 2)
        kk = k[bi].to(torch.float64).repeat_interleave(2, dim=1).permute(1, 0, 2)
        vv = v[bi].to(torch.float64).repeat_interleave(2, dim=1).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, kk, vv, attn_mask=mask[None], scale=scale).permute(1, 0, 2).numpy()
        rows = mask.any(dim=1).numpy()
        np.testing.assert_allclose(out[bi][rows], ref[rows], rtol=0, atol=1e-12)


def test_tiny_workload_matches_brute_force_one_group():
    w = workload.WORKLOADS["tiny"]
    x = workload.make(w)
    # heads 0 and 1 form kv group 0; brute force one group (the blocked oracle
    # runs all heads) to keep the pure-Python loop within seconds.
    out, lse = A.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], x["ids"], x["pos"],
                          w.window_left, w.scale)
    qs = x["q"][:, :, 0:2]
    bo, bl = brute.attn_fwd(_nested(qs), _nested(x["k"][:, :, 0:1]), _nested(x["v"][:, :, 0:1]),
                            x["ids"].tolist(), x["pos"].tolist(), x["ids"].tolist(),
                            x["pos"].tolist(), w.window_left, w.scale)
    np.testing.assert_allclose(out[:, :, 0:2], np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[:, 0:2], np.array(bl), rtol=0, atol=1e-12)


def test_matches_torch_sdpa_fp64():
    """Library routine: SDPA with a boolean mask, rows with >= 1 visible key."""
    q, k, v, ids, pos = _small(11, b=2, s=96, hq=6, hkv=3, d=16, random_pack=True)
    scale = 0.3
    out, lse = A.attn_fwd(q, k, v, ids, pos, ids, pos, 17, scale)
    g = 2
    for bi in range(2):
        mask = torch.from_numpy(A.visible(ids[bi].numpy(), pos[bi].numpy(),
                                          ids[bi].numpy(), pos[bi].numpy(), 17))
        qq = q[bi].to(torch.float64).permute(1, 0, 2)
        kk = k[bi].to(torch.float64).repeat_interleave(g, dim=1).permute(1, 0, 2)
        vv = v[bi].to(torch.float64).repeat_interleave(g, dim=1).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, kk, vv, attn_mask=mask[None], scale=scale).permute(1, 0, 2).numpy()
        rows = mask.any(dim=1).numpy()
        np.testing.assert_allclose(out[bi][rows], ref[rows], rtol=0, atol=1e-12)
        s = torch.einsum("hid,hjd->hij", qq, kk) * scale
        s = s.masked_fill(~mask[None], -math.inf)
        ref_lse = torch.logsumexp(s, dim=-1).numpy()
        np.testing.assert_allclose(lse[bi][:, rows], ref_lse[:, rows], rtol=0, atol=1e-12)


def test_zero_query_closed_form():
    """q = 0: uniform weights over the visible keys, LSE = ln(count)."""
    _, k, v, ids, pos = _small(12, b=2, s=64, random_pack=True)
    q = torch.zeros(2, 64, 4, 8)
    out, lse = A.attn_fwd(q, k, v, ids, pos, ids, pos, 9, 0.5)
    vv = v.to(torch.float64).numpy()
    for bi in range(2):
        m = A.visible(ids[bi].numpy(), pos[bi].numpy(), ids[bi].numpy(), pos[bi].numpy(), 9)
        cnt = m.sum(1)
        for h in range(4):
            for i in range(64):
                if cnt[i] == 0:
                    assert lse[bi, h, i] == -np.inf
                    continue
                ref = vv[bi, m[i], h // 2, :].mean(axis=0)
                np.testing.assert_allclose(out[bi, i, h], ref, atol=1e-13)
                assert abs(lse[bi, h, i] - math.log(cnt[i])) < 1e-13


def test_constant_value_gives_constant_output_and_rows_sum_to_one():
    q, k, _, ids, pos = _small(13, b=1, s=80, random_pack=True)
    v = torch.full((1, 80, 2, 8), 0.0)
    v[..., 3] = 1.0  # the output's column 3 is then the row sum of P
    v[..., 5] = -2.5
    out, lse = A.attn_fwd(q, k, v, ids, pos, ids, pos, -1, 0.35)
    rows = np.isfinite(lse[0, 0])
    np.testing.assert_allclose(out[0, rows, :, 3], 1.0, atol=1e-12)
    np.testing.assert_allclose(out[0, rows, :, 5], -2.5, atol=1e-12)
    assert np.all(out[0, ~rows] == 0.0)


def test_gqa_equals_mha_with_repeated_kv():
    q, k, v, ids, pos = _small(14, b=1, s=48, hq=8, hkv=2, d=8, random_pack=True)
    out, lse = A.attn_fwd(q, k, v, ids, pos, ids, pos, 6, 0.4)
    kr = k.repeat_interleave(4, dim=2)
    vr = v.repeat_interleave(4, dim=2)
    out2, lse2 = A.attn_fwd(q, kr, vr, ids, pos, ids, pos, 6, 0.4)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_wide_window_is_plain_causal():
    q, k, v, ids, pos = _small(15, s=64, slots=2)
    a = A.attn_fwd(q, k, v, ids, pos, ids, pos, -1, 0.3)
    b = A.attn_fwd(q, k, v, ids, pos, ids, pos, 64, 0.3)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    c = A.attn_fwd(q, k, v, ids, pos, ids, pos, 3, 0.3)
    assert not np.allclose(a[0], c[0])


def test_segment_isolation():
    """Perturbing one segment's tokens leaves every other segment unchanged."""
    q, k, v, ids, pos = _small(16, s=64, slots=4)
    base = A.attn_fwd(q, k, v, ids, pos, ids, pos, -1, 0.3)
    sel = (ids[0] == 2)
    k2, v2, q2 = k.clone(), v.clone(), q.clone()
    k2[0, sel] += 1.0
    v2[0, sel] -= 3.0
    q2[0, sel] *= 2.0
    pert = A.attn_fwd(q2, k2, v2, ids, pos, ids, pos, -1, 0.3)
    keep = ~sel.numpy()
    np.testing.assert_array_equal(base[0][0, keep], pert[0][0, keep])
    assert not np.allclose(base[0][0, sel.numpy()], pert[0][0, sel.numpy()])


def test_padding_rows_are_zero_and_neg_inf():
    w = workload.WORKLOADS["packed_thd"]
    s = 512
    q, k, v = workload.qkv(1, s, 2, 1, 8, seed=3)
    ids, pos = workload.segments(1, s, 4)
    out, lse = A.attn_fwd(q, k, v, ids, pos, ids, pos, w.window_left, 0.3)
    pad = (ids[0] == 0).numpy()
    assert pad.sum() == 4 * 32
    assert np.all(out[0, pad] == 0.0)
    assert np.all(np.isneginf(lse[0][:, pad]))
    assert np.all(np.isfinite(lse[0][:, ~pad]))


def _closed_form_pairs(valid_len, window):
    """Visible pairs of one segment of valid_len tokens (inclusive window)."""
    if window < 0 or window >= valid_len - 1:
        return valid_len * (valid_len + 1) // 2
    return (window + 1) * (window + 2) // 2 + (valid_len - window - 1) * (window + 1)


@pytest.mark.parametrize("name", ["tiny", "packed_thd", "packed_swa", "ring_cp4", "full_swa_64k"])
def test_pair_count_closed_form(name):
    w = workload.WORKLOADS[name]
    ids, pos = workload.segments(w.b, w.s, w.slots)
    n_seg = 1 if w.slots is None else w.slots
    valid = w.s if w.slots is None else 3 * (w.s // w.slots) // 4
    expect = w.b * n_seg * _closed_form_pairs(valid, w.window_left)
    got = sum(A.count_pairs(ids[bi], pos[bi], ids[bi], pos[bi], w.window_left) for bi in range(w.b))
    assert got == expect


def test_pair_count_matches_mask_popcount():
    ids, pos = workload.random_segments(2, 300, seed=21)
    for win in (-1, 0, 5, 40):
        for bi in range(2):
            m = A.visible(ids[bi].numpy(), pos[bi].numpy(), ids[bi].numpy(), pos[bi].numpy(), win)
            assert A.count_pairs(ids[bi], pos[bi], ids[bi], pos[bi], win) == int(m.sum())


def test_workload_matches_tutorial_constants():
    with open(os.path.join(GOLDEN, "tutorial_workload.json")) as f:
        gold = json.load(f)
    w = workload.WORKLOADS["full_swa_64k"]
    assert (w.b, w.s, w.hq, w.hkv, w.d) == (gold["batch"], gold["seq"], gold["num_query_heads"],
                                            gold["num_kv_heads"], gold["head_dim"])
    assert w.slots == gold["segments_per_seq"]
    assert [w.window_left, 0] == gold["window_size"]
    assert workload.SEED == gold["seed"]
    ids, pos = workload.segments(w.b, w.s, w.slots)
    slot = gold["slot_len"]
    for sl in range(w.slots):
        seg = ids[0, sl * slot:(sl + 1) * slot]
        assert int((seg == sl + 1).sum()) == gold["valid_tokens_per_slot"]
        assert int((seg == 0).sum()) == gold["padding_tokens_per_slot"]
        assert torch.equal(pos[0, sl * slot:(sl + 1) * slot], torch.arange(slot, dtype=torch.int32))
    assert torch.equal(ids[0], ids[1])
