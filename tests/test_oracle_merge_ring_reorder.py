"""Pins for the merge, reorder, ring and plan oracles (CPU only)."""
import itertools

import numpy as np
import pytest
import torch

import workload
from oracle import attention as A
from oracle import merge as M
from oracle import plan as PL
from oracle import reorder as RO
from oracle import ring as RG


def test_merge_over_any_key_split_equals_one_shot_softmax():
    rng = np.random.default_rng(0)
    n, r, d = 50, 7, 5
    scores = rng.normal(size=(r, n)) * 4
    vis = rng.random((r, n)) < 0.6
    vis[3] = False  # one row with no visible key
    vals = rng.normal(size=(n, d))
    s = np.where(vis, scores, -np.inf)
    has = vis.any(1)
    p = np.where(vis, np.exp(s - np.where(has, s.max(1), 0)[:, None]), 0)
    z = p.sum(1)
    ref = np.where(has[:, None], (p / np.where(has, z, 1)[:, None]) @ vals, 0)
    cuts = [0, 9, 10, 23, 40, 50]
    blocks = [slice(a, b) for a, b in zip(cuts[:-1], cuts[1:])]
    for order in itertools.permutations(range(len(blocks))):
        m, zz, u = np.full(r, -np.inf), np.zeros(r), np.zeros((r, d))
        for bidx in order:
            bl = blocks[bidx]
            mb, zb, ub = M.block_stats(scores[:, bl], vis[:, bl], vals[bl])
            m, zz, u = M.merge_mzu(m, zz, u, mb, zb, ub)
        out, lse = M.finish(m, zz, u)
        np.testing.assert_allclose(out, ref, atol=1e-12)
        assert np.isneginf(lse[3]) and np.all(out[3] == 0)


def test_merge_partial_of_key_halves_equals_full_attention():
    q, k, v = workload.qkv(2, 64, 4, 2, 8, seed=5)
    ids, pos = workload.random_segments(2, 64, seed=5)
    full = A.attn_fwd(q, k, v, ids, pos, ids, pos, 11, 0.3)
    # keys split into two halves: attention of every query over each half
    halves = []
    for lo, hi in ((0, 30), (30, 64)):
        halves.append(A.attn_fwd(q, k[:, lo:hi], v[:, lo:hi], ids, pos, ids[:, lo:hi],
                                 pos[:, lo:hi], 11, 0.3))
    for order in ((0, 1), (1, 0)):
        o, l = M.merge_partial(halves[order[0]][0], halves[order[0]][1],
                               halves[order[1]][0], halves[order[1]][1])
        np.testing.assert_allclose(o, full[0], atol=1e-12)
        assert np.array_equal(np.isneginf(l), np.isneginf(full[1]))
        fin = np.isfinite(full[1])
        np.testing.assert_allclose(l[fin], full[1][fin], atol=1e-12)


def test_separate_softmax_per_block_is_wrong():
    """The pages warn against normalising each remote block on its own: the
    merge must not equal a plain average of per-block outputs."""
    q, k, v = workload.qkv(1, 32, 2, 1, 4, seed=9)
    ids = torch.ones(1, 32, dtype=torch.int32)
    pos = torch.arange(32, dtype=torch.int32)[None]
    full = A.attn_fwd(q, k, v, ids, pos, ids, pos, -1, 0.5)
    a = A.attn_fwd(q, k[:, :16], v[:, :16], ids, pos, ids[:, :16], pos[:, :16], -1, 0.5)
    b = A.attn_fwd(q, k[:, 16:], v[:, 16:], ids, pos, ids[:, 16:], pos[:, 16:], -1, 0.5)
    rows = slice(16, 32)
    naive = 0.5 * (a[0] + b[0])
    assert not np.allclose(naive[:, rows], full[0][:, rows], atol=1e-3)
    o, _ = M.merge_partial(a[0], a[1], b[0], b[1])
    np.testing.assert_allclose(o, full[0], atol=1e-12)


def test_dual_chunk_small_example():
    # s = 8, R = 2: chunks of 2; shard 0 = chunks 0 and 3, shard 1 = chunks 1 and 2
    assert RO.dual_chunk_src(8, 2).tolist() == [0, 1, 6, 7, 2, 3, 4, 5]
    # s = 16, R = 4: chunks of 2; shard r = chunks r and 7 - r
    assert RO.dual_chunk_src(16, 4).tolist() == [0, 1, 14, 15, 2, 3, 12, 13, 4, 5, 10, 11,
                                                 6, 7, 8, 9]


def test_striped_small_example():
    # stripes of 2 over R = 2: stripes 0,2 -> shard 0, stripes 1,3 -> shard 1
    assert RO.striped_src(8, 2, 2).tolist() == [0, 1, 4, 5, 2, 3, 6, 7]
    assert RO.striped_src(8, 4, 1).tolist() == [0, 4, 1, 5, 2, 6, 3, 7]


@pytest.mark.parametrize("strategy,R,stripe,s", [
    (RO.DUAL_CHUNK, 4, 1, 32768), (RO.DUAL_CHUNK, 2, 1, 24), (RO.STRIPED, 4, 1, 4096),
    (RO.STRIPED, 4, 512, 65536), (RO.STRIPED, 3, 2, 36)])
def test_reorder_is_bijection_and_inverse_is_identity(strategy, R, stripe, s):
    src = RO.src_index(s, strategy, R, stripe)
    assert np.array_equal(np.sort(src), np.arange(s))
    x = np.arange(2 * s * 3).reshape(2, s, 3)
    y = RO.reorder(x, strategy, R, stripe)
    assert np.array_equal(RO.inverse_reorder(y, strategy, R, stripe), x)
    assert np.array_equal(y[:, :, 0] // 3 % s, np.broadcast_to(src, (2, s)))


def test_dual_chunk_balances_causal_work():
    """Each shard's causal work (sum of positions + 1 of its queries) is equal."""
    s, R = 64, 4
    src = RO.dual_chunk_src(s, R)
    n = s // R
    work = [int((src[r * n:(r + 1) * n] + 1).sum()) for r in range(R)]
    assert len(set(work)) == 1


@pytest.mark.parametrize("seed,window,R,strategy,stripe,pack", [
    (1, -1, 4, RO.DUAL_CHUNK, 1, None), (2, 7, 2, RO.DUAL_CHUNK, 1, 2),
    (3, -1, 4, RO.STRIPED, 1, 4), (4, 5, 2, RO.STRIPED, 4, None)])
def test_ring_emulation_equals_full_attention(seed, window, R, strategy, stripe, pack):
    s = 64
    q, k, v = workload.qkv(1, s, 4, 2, 8, seed=seed)
    ids, pos = workload.segments(1, s, pack)
    full = A.attn_fwd(q, k, v, ids, pos, ids, pos, window, 0.35)
    o, l = RG.ring_attention(q, k, v, ids, pos, window, 0.35, R, strategy, stripe)
    np.testing.assert_allclose(o, full[0], atol=1e-12)
    assert np.array_equal(np.isneginf(l), np.isneginf(full[1]))
    fin = np.isfinite(full[1])
    np.testing.assert_allclose(l[fin], full[1][fin], atol=1e-12)


def test_ring_without_position_mask_would_differ():
    """Masking by reordered array index instead of segment position breaks
    causality across shard boundaries: the ring oracle must not do that."""
    s = 32
    q, k, v = workload.qkv(1, s, 2, 1, 4, seed=8)
    ids, pos = workload.segments(1, s, None)
    src = RO.dual_chunk_src(s, 2)
    wrong_pos = torch.arange(s, dtype=torch.int32)[None]  # index, not position
    qr, kr, vr = q[:, src], k[:, src], v[:, src]
    bad = A.attn_fwd(qr, kr, vr, ids, wrong_pos, ids, wrong_pos, -1, 0.5)[0]
    good = RO.inverse_reorder(bad, RO.DUAL_CHUNK, 2)
    full = A.attn_fwd(q, k, v, ids, pos, ids, pos, -1, 0.5)[0]
    assert not np.allclose(good, full)
    o, _ = RG.ring_attention(q, k, v, ids, pos, -1, 0.5, 2)
    np.testing.assert_allclose(o, full, atol=1e-12)


def _plan_case(ids, pos, window, tile):
    cls = PL.classes(ids, pos, ids, pos, window, tile)
    exact = PL.brute_classes(ids, pos, ids, pos, window, tile)
    # never skip a visible pair, never call a tile with an invisible pair FULL
    assert not np.any((cls == PL.SKIP) & (exact != PL.SKIP))
    assert not np.any((cls == PL.FULL) & (exact != PL.FULL))
    # the pair count rebuilt from the plan equals the brute-force count
    b = ids.shape[0]
    total = 0
    for bi in range(b):
        m = A.visible(ids[bi], pos[bi], ids[bi], pos[bi], window)
        s = m.shape[0]
        for a in range(cls.shape[1]):
            for c in range(cls.shape[2]):
                blk = m[a * tile:(a + 1) * tile, c * tile:(c + 1) * tile]
                if cls[bi, a, c] == PL.FULL:
                    total += blk.size
                elif cls[bi, a, c] == PL.PARTIAL:
                    total += int(blk.sum())
        assert s == ids.shape[1]
    want = sum(A.count_pairs(ids[bi], pos[bi], ids[bi], pos[bi], window) for bi in range(b))
    assert total == want
    return cls, exact


@pytest.mark.parametrize("window", [-1, 0, 100, 300])
def test_plan_is_safe_on_random_packing(window):
    ids, pos = workload.random_segments(2, 1000, seed=31 + window)
    _plan_case(ids.numpy(), pos.numpy(), window, 128)


@pytest.mark.parametrize("s,slots,window,tile", [
    (4096, 4, -1, 128), (4096, 4, 1024, 128), (2048, None, -1, 128), (1100, None, 300, 128)])
def test_plan_is_exact_on_tutorial_packing(s, slots, window, tile):
    ids, pos = workload.segments(1, s, slots)
    cls, exact = _plan_case(ids.numpy(), pos.numpy(), window, tile)
    if s % tile == 0:
        assert np.array_equal(cls, exact)


def test_plan_ranges():
    ids, pos = workload.segments(1, 1024, 2)
    cls = PL.classes(ids.numpy(), pos.numpy(), ids.numpy(), pos.numpy(), 200, 128)
    rng = PL.ranges(cls)
    # slot 0 = tokens 0..511 (384 valid = tiles 0..2), tile 3 is padding
    assert tuple(rng[0, 0]) == (0, 0)
    assert tuple(rng[0, 2]) == (0, 2)
    assert tuple(rng[0, 3]) == (0, -1)
    assert tuple(rng[0, 6]) == (4, 6)
