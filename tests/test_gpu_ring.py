"""Ring emulation on one GPU (reorder -> per-step attn_fwd + merge -> inverse
reorder) must equal full attention and the CPU oracle's ring."""
import numpy as np
import pytest
import torch

import workload
from oracle import attention as A
from oracle import reorder as RO
from oracle import ring as RG
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ring():
    from long_context_attention_attn_gb300 import ring as mod
    return mod


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("b,s,hq,hkv,d,window,slots,R,strategy,stripe", [
    (1, 2048, 4, 2, 128, -1, None, 4, RO.DUAL_CHUNK, 1),
    (2, 1536, 4, 1, 64, 200, 2, 3, RO.DUAL_CHUNK, 1),
    (1, 4096, 2, 1, 128, -1, 4, 4, RO.STRIPED, 128),
    (1, 1024, 2, 2, 128, 100, None, 2, RO.STRIPED, 1),
])
def test_ring_matches_oracle(ring, b, s, hq, hkv, d, window, slots, R, strategy, stripe, fused):
    q, k, v = workload.qkv(b, s, hq, hkv, d, seed=R + s)
    ids, pos = workload.segments(b, s, slots)
    out, lse = ring.ring_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), ids.to(DEV), pos.to(DEV), R,
                                  window_left=window, scale=d ** -0.5, strategy=strategy,
                                  stripe_size=stripe, fused_merge=fused)
    torch.cuda.synchronize()
    ro, rl = RG.ring_attention(q, k, v, ids, pos, window, d ** -0.5, R, strategy, stripe)
    check_out(out.cpu(), ro)
    check_lse(lse.cpu(), rl)
    fo, fl = A.attn_fwd(q, k, v, ids, pos, ids, pos, window, d ** -0.5)
    np.testing.assert_allclose(ro, fo, atol=1e-12)


@pytest.mark.parametrize("s,window,slots,R,strategy,stripe", [
    (4096, -1, 4, 4, RO.STRIPED, 512),
    (2048, 300, None, 4, RO.STRIPED, 1),
    (3072, -1, 2, 3, RO.DUAL_CHUNK, 1),
])
def test_allgather_matches_oracle(ring, s, window, slots, R, strategy, stripe):
    q, k, v = workload.qkv(1, s, 4, 2, 128, seed=s + R)
    ids, pos = workload.segments(1, s, slots)
    out, lse = ring.allgather_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), ids.to(DEV), pos.to(DEV),
                                       R, window_left=window, scale=0.0884, strategy=strategy,
                                       stripe_size=stripe)
    torch.cuda.synchronize()
    ro, rl = A.attn_fwd(q, k, v, ids, pos, ids, pos, window, 0.0884)
    check_out(out.cpu(), ro)
    check_lse(lse.cpu(), rl)


def test_allgather_tutorial_shape_sampled(ring):
    """P1's AllGather case: stripe 512 over 4 shards on the 64k packed workload
    (sampled rows against the oracle)."""
    w = workload.WORKLOADS["full_swa_64k"]
    x = workload.make(w, device=DEV, with_dout=False)
    out, lse = ring.allgather_attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], 4,
                                       window_left=w.window_left, scale=w.scale)
    torch.cuda.synchronize()
    ids, pos = x["ids"].cpu(), x["pos"].cpu()
    for bi, h, r0, nr in ((0, 5, 12000, 96), (1, 100, 2 * 16384 + 700, 64)):
        kvh = h // (w.hq // w.hkv)
        rows = np.arange(r0, r0 + nr)
        ro, rl = A.attn_fwd(x["q"][bi:bi + 1, :, h:h + 1].cpu(), x["k"][bi:bi + 1, :, kvh:kvh + 1].cpu(),
                            x["v"][bi:bi + 1, :, kvh:kvh + 1].cpu(), ids[bi:bi + 1], pos[bi:bi + 1],
                            ids[bi:bi + 1], pos[bi:bi + 1], w.window_left, w.scale, rows=rows)
        check_out(out[bi, r0:r0 + nr, h].cpu(), ro[0, rows, 0])
        check_lse(lse[bi, h, r0:r0 + nr].cpu(), rl[0, 0, rows])
    del x, out, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("b,s,hq,hkv,d,window,slots,R,strategy,stripe", [
    (1, 2048, 4, 2, 128, -1, None, 4, RO.DUAL_CHUNK, 1),
    (2, 1536, 4, 1, 64, 200, 2, 3, RO.DUAL_CHUNK, 1),
    (1, 4096, 2, 1, 128, 700, 4, 4, RO.STRIPED, 128),
])
def test_ring_backward_matches_oracle(ring, b, s, hq, hkv, d, window, slots, R, strategy, stripe):
    """Ring-emulated backward (per-block contributions with the final LSE/D,
    fp32 accumulation) equals the oracle's full backward."""
    from tests.parity import check_grad
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=R * 7 + s, with_dout=True)
    ids, pos = workload.segments(b, s, slots)
    g = [x.to(DEV) for x in (q, k, v, dout, ids, pos)]
    out, lse = ring.ring_attn_fwd(g[0], g[1], g[2], g[4], g[5], R, window_left=window,
                                  scale=d ** -0.5, strategy=strategy, stripe_size=stripe)
    dq, dk, dv = ring.ring_attn_bwd(g[0], g[1], g[2], out, lse, g[3], g[4], g[5], R,
                                    window_left=window, scale=d ** -0.5, strategy=strategy,
                                    stripe_size=stripe)
    torch.cuda.synchronize()
    rq, rk, rv = A.attn_bwd(q, k, v, dout, ids, pos, ids, pos, window, d ** -0.5)
    check_grad(dq.cpu(), rq, "dq")
    check_grad(dk.cpu(), rk, "dk")
    check_grad(dv.cpu(), rv, "dv")
    pad = (ids == 0).to(DEV)
    assert torch.all(dq[pad] == 0) and torch.all(dk[pad] == 0) and torch.all(dv[pad] == 0)


def test_ring_workload_equals_full_attention(ring):
    """The 32k ring workload: R = 4 dual-chunk shards, compared with the
    single-call forward on every element and with the oracle on samples."""
    import long_context_attention_attn_gb300 as ga
    w = workload.WORKLOADS["ring_cp4"]
    x = workload.make(w, device=DEV, with_dout=False)
    out, lse = ring.ring_attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], w.cp_size,
                                  window_left=w.window_left, scale=w.scale)
    full_o, full_l = ga.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"],
                                 window_left=w.window_left, scale=w.scale)
    torch.cuda.synchronize()
    # ring vs one-shot GPU forward: both within bf16 rounding of each other
    diff = (out.float() - full_o.float()).abs().max().item()
    assert diff <= 2e-2, diff
    assert (lse - full_l).abs().max().item() <= 1e-3
    ids, pos = x["ids"].cpu(), x["pos"].cpu()
    for h, r0, nr in ((0, 0, 128), (37, 20000, 64), (63, 32768 - 100, 100)):
        kvh = h // (w.hq // w.hkv)
        rows = np.arange(r0, r0 + nr)
        ro, rl = A.attn_fwd(x["q"][:, :, h:h + 1].cpu(), x["k"][:, :, kvh:kvh + 1].cpu(),
                            x["v"][:, :, kvh:kvh + 1].cpu(), ids, pos, ids, pos, w.window_left,
                            w.scale, rows=rows)
        check_out(out[0, r0:r0 + nr, h].cpu(), ro[0, rows, 0])
        check_lse(lse[0, h, r0:r0 + nr].cpu(), rl[0, 0, rows])


@pytest.mark.parametrize("final", [False, True])
def test_fwd_merge_mode_matches_oracle_merge(final):
    """attn_fwd with merge_into_out folds a block into an accumulator exactly
    like the oracle's merge of the two partials; rows whose accumulator is
    empty (LSE -inf, out holding NaN) take the block, rows seeing no key in
    either keep (0, -inf)."""
    import long_context_attention_attn_gb300 as ga
    from oracle import merge as MG
    b, s, hq, hkv, d = 1, 640, 4, 2, 128
    q, k, v = workload.qkv(b, 2 * s, hq, hkv, d, seed=77)
    ids, pos = workload.segments(b, 2 * s, None)
    ids[:, 600:700] = 0  # padding rows and keys inside both halves
    qa, ia, pa = q[:, s:], ids[:, s:], pos[:, s:]
    # accumulator: the second half's queries against the first half's keys
    acc_o, acc_l = A.attn_fwd(qa, k[:, :s], v[:, :s], ia, pa, ids[:, :s], pos[:, :s], -1, d ** -0.5)
    blk_o, blk_l = A.attn_fwd(qa, k[:, s:], v[:, s:], ia, pa, ids[:, s:], pos[:, s:], -1, d ** -0.5)
    want_o, want_l = MG.merge_partial(acc_o, acc_l, blk_o, blk_l)
    acc = torch.from_numpy(acc_o).float().to(DEV)
    lacc = torch.from_numpy(acc_l).float().to(DEV)
    acc[torch.isinf(lacc).transpose(1, 2).unsqueeze(-1).expand_as(acc)] = float("nan")
    fin = torch.empty(b, s, hq, d, dtype=torch.bfloat16, device=DEV) if final else None
    ga.attn_fwd(qa.to(DEV), k[:, s:].to(DEV), v[:, s:].to(DEV), ia.to(DEV), pa.to(DEV),
                ids[:, s:].to(DEV), pos[:, s:].to(DEV), scale=d ** -0.5, out=acc, lse=lacc,
                out_fp32=True, merge_into_out=True, out_final=fin)
    torch.cuda.synchronize()
    check_out((fin if final else acc).float().cpu(), want_o)
    check_lse(lacc.cpu(), want_l)


def test_ring_backward_at_ring_workload(ring):
    """The 32k ring workload's backward as R = 4 dual-chunk ring shards
    (per-block attn_bwd, fp32 accumulation with the final LSE): equal to the
    single-call backward on every element (both within the gradient
    tolerance of each other) and to the oracle on sampled query rows (dQ) and
    key tiles (dK, dV, complete: every row that sees those keys is included)."""
    import long_context_attention_attn_gb300 as ga
    from tests.parity import check_grad
    w = workload.WORKLOADS["ring_cp4"]
    x = workload.make(w, device=DEV, with_dout=True)
    q, k, v, ids, pos, dout = x["q"], x["k"], x["v"], x["ids"], x["pos"], x["dout"]
    out, lse = ga.attn_fwd(q, k, v, ids, pos, window_left=w.window_left, scale=w.scale)
    dq, dk, dv = ring.ring_attn_bwd(q, k, v, out, lse, dout, ids, pos, w.cp_size,
                                    window_left=w.window_left, scale=w.scale)
    fq, fk, fv = ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, window_left=w.window_left,
                             scale=w.scale)
    torch.cuda.synchronize()
    for name, a_, b_ in (("dq", dq, fq), ("dk", dk, fk), ("dv", dv, fv)):
        num = (a_.float() - b_.float()).norm().item()
        den = b_.float().norm().item()
        assert num <= 1e-2 * den, f"ring vs single-call {name}: rel-L2 {num / den:.3e}"
    g = w.hq // w.hkv
    idc, psc = ids.cpu(), pos.cpu()
    for kvh, r0, nr in ((0, 0, 128), (4, 20000, 64), (7, 32768 - 96, 96)):
        hs = slice(kvh * g, kvh * g + g)
        rows = np.arange(r0, r0 + nr)
        rq, _, _ = A.attn_bwd(q[:, :, hs].cpu(), k[:, :, kvh:kvh + 1].cpu(),
                              v[:, :, kvh:kvh + 1].cpu(), dout[:, :, hs].cpu(), idc, psc, idc,
                              psc, w.window_left, w.scale, rows=rows)
        check_grad(dq[0, r0:r0 + nr, hs].cpu(), rq[0, rows], f"dq kvh{kvh} r{r0}")
    for kvh, k0, nk in ((2, 32768 - 128, 128), (6, 32768 - 200, 72)):
        keys = np.arange(k0, k0 + nk)
        rows = A.rows_seeing_keys(idc[0], psc[0], idc[0], psc[0], w.window_left, keys)
        hs = slice(kvh * g, kvh * g + g)
        _, rk, rv = A.attn_bwd(q[:, :, hs].cpu(), k[:, :, kvh:kvh + 1].cpu(),
                               v[:, :, kvh:kvh + 1].cpu(), dout[:, :, hs].cpu(), idc, psc, idc,
                               psc, w.window_left, w.scale, rows=rows)
        check_grad(dk[0, k0:k0 + nk, kvh].cpu(), rk[0, keys, 0], f"dk kvh{kvh} k{k0}")
        check_grad(dv[0, k0:k0 + nk, kvh].cpu(), rv[0, keys, 0], f"dv kvh{kvh} k{k0}")


def test_ring_backward_deterministic_mode(ring):
    """ring_attn_bwd(deterministic=True): every block call sums its dQ on chip
    in a fixed order, so two runs give the same bits, and the result equals
    the oracle's full backward."""
    from tests.parity import check_grad
    b, s, hq, hkv, d, window, R = 1, 2048, 4, 2, 128, 700, 4
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=91, with_dout=True)
    ids, pos = workload.segments(b, s, 2)
    g = [x.to(DEV) for x in (q, k, v, dout, ids, pos)]
    out, lse = ring.ring_attn_fwd(g[0], g[1], g[2], g[4], g[5], R, window_left=window,
                                  scale=d ** -0.5)
    runs = [ring.ring_attn_bwd(g[0], g[1], g[2], out, lse, g[3], g[4], g[5], R,
                               window_left=window, scale=d ** -0.5, deterministic=True)
            for _ in range(2)]
    torch.cuda.synchronize()
    for a_, b_ in zip(*runs):
        assert torch.equal(a_, b_)
    rq, rk, rv = A.attn_bwd(q, k, v, dout, ids, pos, ids, pos, window, d ** -0.5)
    check_grad(runs[0][0].cpu(), rq, "dq")
    check_grad(runs[0][1].cpu(), rk, "dk")
    check_grad(runs[0][2].cpu(), rv, "dv")


@pytest.mark.parametrize("b,s,hq,hkv,d,window,slots,R,strategy,stripe", [
    (1, 4096, 4, 2, 128, -1, 4, 4, RO.STRIPED, 512),
    (2, 2048, 4, 1, 64, 300, 2, 4, RO.STRIPED, 128),
    (1, 3072, 2, 2, 128, -1, None, 3, RO.DUAL_CHUNK, 1),
])
def test_allgather_backward_matches_oracle(ring, b, s, hq, hkv, d, window, slots, R, strategy,
                                           stripe):
    """All-gather backward: each shard's queries against the whole reordered
    K/V in one attn_bwd call, dK/dV summed over the shards in fp32; equals the
    oracle's full backward, with exact zeros on padding."""
    from tests.parity import check_grad
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=R * 11 + s, with_dout=True)
    ids, pos = workload.segments(b, s, slots)
    g = [x.to(DEV) for x in (q, k, v, dout, ids, pos)]
    out, lse = ring.allgather_attn_fwd(g[0], g[1], g[2], g[4], g[5], R, window_left=window,
                                       scale=d ** -0.5, strategy=strategy, stripe_size=stripe)
    dq, dk, dv = ring.allgather_attn_bwd(g[0], g[1], g[2], out, lse, g[3], g[4], g[5], R,
                                         window_left=window, scale=d ** -0.5, strategy=strategy,
                                         stripe_size=stripe)
    torch.cuda.synchronize()
    rq, rk, rv = A.attn_bwd(q, k, v, dout, ids, pos, ids, pos, window, d ** -0.5)
    check_grad(dq.cpu(), rq, "dq")
    check_grad(dk.cpu(), rk, "dk")
    check_grad(dv.cpu(), rv, "dv")
    pad = (ids == 0).to(DEV)
    assert torch.all(dq[pad] == 0) and torch.all(dk[pad] == 0) and torch.all(dv[pad] == 0)


def test_allgather_backward_tutorial_shape(ring):
    """The TE tutorial's AllGather case (64k packed workload, 4 shards, stripe
    512) backward: equal to the single-call backward on every element (both
    within the gradient tolerance of each other) and to the oracle on sampled
    query rows (dQ) and key tiles (dK, dV, complete: every row that sees those
    keys is included)."""
    import long_context_attention_attn_gb300 as ga
    from tests.parity import check_grad
    w = workload.WORKLOADS["full_swa_64k"]
    x = workload.make(w, device=DEV, with_dout=True)
    q, k, v, ids, pos, dout = x["q"], x["k"], x["v"], x["ids"], x["pos"], x["dout"]
    out, lse = ga.attn_fwd(q, k, v, ids, pos, window_left=w.window_left, scale=w.scale)
    dq, dk, dv = ring.allgather_attn_bwd(q, k, v, out, lse, dout, ids, pos, 4,
                                         window_left=w.window_left, scale=w.scale)
    fq, fk, fv = ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, window_left=w.window_left,
                             scale=w.scale)
    torch.cuda.synchronize()
    for name, a_, b_ in (("dq", dq, fq), ("dk", dk, fk), ("dv", dv, fv)):
        num = (a_.float() - b_.float()).norm().item()
        den = b_.float().norm().item()
        assert num <= 1e-2 * den, f"all-gather vs single-call {name}: rel-L2 {num / den:.3e}"
    del fq, fk, fv
    g = w.hq // w.hkv
    idc, psc = ids.cpu(), pos.cpu()
    for bi, kvh, r0, nr in ((0, 1, 9000, 64), (1, 6, 3 * 16384 + 5000, 64)):
        hs = slice(kvh * g, kvh * g + g)
        rows = np.arange(r0, r0 + nr)
        rq, _, _ = A.attn_bwd(q[bi:bi + 1, :, hs].cpu(), k[bi:bi + 1, :, kvh:kvh + 1].cpu(),
                              v[bi:bi + 1, :, kvh:kvh + 1].cpu(), dout[bi:bi + 1, :, hs].cpu(),
                              idc[bi:bi + 1], psc[bi:bi + 1], idc[bi:bi + 1], psc[bi:bi + 1],
                              w.window_left, w.scale, rows=rows)
        check_grad(dq[bi, r0:r0 + nr, hs].cpu(), rq[0, rows], f"dq b{bi} kvh{kvh} r{r0}")
    for bi, kvh, k0, nk in ((0, 3, 16384 + 11000, 64),):
        keys = np.arange(k0, k0 + nk)
        rows = A.rows_seeing_keys(idc[bi], psc[bi], idc[bi], psc[bi], w.window_left, keys)
        hs = slice(kvh * g, kvh * g + g)
        _, rk, rv = A.attn_bwd(q[bi:bi + 1, :, hs].cpu(), k[bi:bi + 1, :, kvh:kvh + 1].cpu(),
                               v[bi:bi + 1, :, kvh:kvh + 1].cpu(), dout[bi:bi + 1, :, hs].cpu(),
                               idc[bi:bi + 1], psc[bi:bi + 1], idc[bi:bi + 1], psc[bi:bi + 1],
                               w.window_left, w.scale, rows=rows)
        check_grad(dk[bi, k0:k0 + nk, kvh].cpu(), rk[0, keys, 0], f"dk b{bi} kvh{kvh} k{k0}")
        check_grad(dv[bi, k0:k0 + nk, kvh].cpu(), rv[0, keys, 0], f"dv b{bi} kvh{kvh} k{k0}")
    del x, out, lse, dq, dk, dv
    torch.cuda.empty_cache()


@pytest.mark.parametrize("b,s,hq,hkv,d,window,slots,R,strategy,stripe", [
    (1, 2048, 4, 2, 128, -1, None, 4, RO.DUAL_CHUNK, 1),
    (2, 1536, 4, 1, 64, 200, 2, 3, RO.DUAL_CHUNK, 1),
    (1, 4096, 2, 1, 128, -1, 4, 4, RO.STRIPED, 128),
])
def test_ring_batched_shards(ring, b, s, hq, hkv, d, window, slots, R, strategy, stripe):
    """batch_shards=True (one call per ring step over all shards, K/V blocks
    and dK / dV sums rotated between steps): the forward equals the per-shard
    form bit for bit (every block computes the same tiles and merges in the
    same step order), the backward equals the oracle (its dK / dV sums over
    the shards run in another order)."""
    from tests.parity import check_grad
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=R * 13 + s, with_dout=True)
    ids, pos = workload.segments(b, s, slots)
    g = [x.to(DEV) for x in (q, k, v, dout, ids, pos)]
    kw = dict(window_left=window, scale=d ** -0.5, strategy=strategy, stripe_size=stripe)
    for fused in (True, False):
        o1, l1 = ring.ring_attn_fwd(g[0], g[1], g[2], g[4], g[5], R, fused_merge=fused, **kw)
        o2, l2 = ring.ring_attn_fwd(g[0], g[1], g[2], g[4], g[5], R, fused_merge=fused,
                                    batch_shards=True, **kw)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    dq, dk, dv = ring.ring_attn_bwd(g[0], g[1], g[2], o1, l1, g[3], g[4], g[5], R,
                                    batch_shards=True, **kw)
    torch.cuda.synchronize()
    rq, rk, rv = A.attn_bwd(q, k, v, dout, ids, pos, ids, pos, window, d ** -0.5)
    check_grad(dq.cpu(), rq, "dq")
    check_grad(dk.cpu(), rk, "dk")
    check_grad(dv.cpu(), rv, "dv")
    pad = (ids == 0).to(DEV)
    assert torch.all(dq[pad] == 0) and torch.all(dk[pad] == 0) and torch.all(dv[pad] == 0)
    # deterministic mode: fixed-order sums, two runs give the same bits
    runs = [ring.ring_attn_bwd(g[0], g[1], g[2], o1, l1, g[3], g[4], g[5], R, batch_shards=True,
                               deterministic=True, **kw) for _ in range(2)]
    torch.cuda.synchronize()
    for a_, b_ in zip(*runs):
        assert torch.equal(a_, b_)
