"""GPU parity of attn_bwd through the C ABI against the CPU oracle.

The oracle differentiates the exact float64 attention itself (its own O for
D = rowsum(dO * O)); the GPU consumes its own bf16 forward output and LSE, as
a training step would.  Small cases are compared on every element; the large
workloads on sampled query rows (dQ) and sampled key tiles (dK, dV, complete
because every query row that sees those keys is included)."""
import numpy as np
import pytest
import torch

import workload
from oracle import attention as A
from tests.parity import check_grad, check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ga():
    import long_context_attention_attn_gb300 as pkg
    return pkg


def _gpu_grads(ga, x, window, scale, det=False):
    g = {k: v.to(DEV) for k, v in x.items()}
    out, lse = ga.attn_fwd(g["q"], g["k"], g["v"], g["ids"], g["pos"], window_left=window,
                           scale=scale)
    dq, dk, dv = ga.attn_bwd(g["q"], g["k"], g["v"], out, lse, g["dout"], g["ids"], g["pos"],
                             window_left=window, scale=scale, deterministic=det,
                             check_status=True)
    torch.cuda.synchronize()
    return dq.cpu(), dk.cpu(), dv.cpu()


def _full_check(ga, x, window, scale, det=False):
    dq, dk, dv = _gpu_grads(ga, x, window, scale, det)
    rq, rk, rv = A.attn_bwd(x["q"], x["k"], x["v"], x["dout"], x["ids"], x["pos"], x["ids"],
                            x["pos"], window, scale)
    check_grad(dq, rq, "dq")
    check_grad(dk, rk, "dk")
    check_grad(dv, rv, "dv")
    pad = (x["ids"] == 0)
    assert torch.all(dq[pad] == 0) and torch.all(dk[pad] == 0) and torch.all(dv[pad] == 0)


@pytest.mark.parametrize("det", [False, True])
def test_tiny_workload(ga, det):
    w = workload.WORKLOADS["tiny"]
    _full_check(ga, workload.make(w, with_dout=True), w.window_left, w.scale, det)


@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("b,s,hq,hkv,d,window,seed", [
    (2, 300, 4, 1, 128, 70, 1),   # ragged tail, g = 4
    (1, 200, 3, 1, 64, -1, 2),    # odd group
    (1, 384, 2, 2, 128, -1, 3),   # g = 1
    (1, 640, 4, 2, 128, 0, 4),    # window 0
    (2, 6000, 2, 1, 128, 700, 5),  # plan above 4096 class bytes: the parallel plan kernels
])
def test_random_packing(ga, b, s, hq, hkv, d, window, seed, det):
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=seed, with_dout=True)
    ids, pos = workload.random_segments(b, s, seed=seed)
    x = dict(q=q, k=k, v=v, dout=dout, ids=ids, pos=pos)
    _full_check(ga, x, window, d ** -0.5, det)


@pytest.mark.parametrize("name", ["packed_swa", "tiny"])
def test_deterministic_mode_is_bit_identical(ga, name):
    """deterministic=True: dQ is summed on chip in a fixed order, so three
    backward calls on the same inputs give the same bits in dq, dk and dv."""
    w = workload.WORKLOADS[name]
    x = workload.make(w, device=DEV, with_dout=True)
    out, lse = ga.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], window_left=w.window_left,
                           scale=w.scale)
    runs = [ga.attn_bwd(x["q"], x["k"], x["v"], out, lse, x["dout"], x["ids"], x["pos"],
                        window_left=w.window_left, scale=w.scale, deterministic=True)
            for _ in range(3)]
    torch.cuda.synchronize()
    for r in runs[1:]:
        for a_, b_ in zip(r, runs[0]):
            assert torch.equal(a_, b_)



@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("s_q,s_kv,q0,window,d,seed", [
    (256, 384, 300, 200, 128, 11),   # queries late in the kv range, window crossing tiles
    (200, 520, 100, -1, 64, 12),     # ragged on both sides, unlimited window
    (384, 130, 0, 40, 128, 13),      # more queries than keys (rows past the keys see none)
])
def test_cross_descriptor_and_lengths(ga, s_q, s_kv, q0, window, d, seed, det):
    """Queries of one shard against keys of another, of a different length
    and with a padding hole in the keys (the per-block call of a ring step
    with its own q and kv descriptors)."""
    hq, hkv = 4, 2
    q, _, _, dout = workload.qkv(1, s_q, hq, hkv, d, seed=seed, with_dout=True)
    _, k, v = workload.qkv(1, s_kv, hq, hkv, d, seed=seed + 100)
    ids = torch.ones(1, s_q, dtype=torch.int32)
    pos = torch.arange(q0, q0 + s_q, dtype=torch.int32)[None]
    kv_ids = torch.ones(1, s_kv, dtype=torch.int32)
    kv_pos = torch.arange(0, s_kv, dtype=torch.int32)[None]
    kv_ids[0, s_kv // 3:s_kv // 3 + 30] = 0
    scale = d ** -0.5
    g = {n: t.to(DEV) for n, t in dict(q=q, k=k, v=v, dout=dout, ids=ids, pos=pos,
                                       kv_ids=kv_ids, kv_pos=kv_pos).items()}
    out, lse = ga.attn_fwd(g["q"], g["k"], g["v"], g["ids"], g["pos"], g["kv_ids"], g["kv_pos"],
                           window_left=window, scale=scale)
    dq, dk, dv = ga.attn_bwd(g["q"], g["k"], g["v"], out, lse, g["dout"], g["ids"], g["pos"],
                             g["kv_ids"], g["kv_pos"], window_left=window, scale=scale,
                             deterministic=det)
    torch.cuda.synchronize()
    rq, rk, rv = A.attn_bwd(q, k, v, dout, ids, pos, kv_ids, kv_pos, window, scale)
    check_grad(dq.cpu(), rq, "dq")
    check_grad(dk.cpu(), rk, "dk")
    check_grad(dv.cpu(), rv, "dv")
    # keys no query can see (padding, or outside every query's window) get exactly 0
    ro, _ = A.attn_fwd(q, k, v, ids, pos, kv_ids, kv_pos, window, scale)
    unseen = torch.from_numpy(np.abs(rk).sum(axis=(2, 3)) == 0)
    assert torch.all(dk.cpu()[unseen] == 0) and torch.all(dv.cpu()[unseen] == 0)
    # query rows that see no key get dQ = 0 exactly
    blind = torch.from_numpy(np.abs(ro).sum(axis=(2, 3)) == 0)
    assert torch.all(dq.cpu()[blind] == 0)


@pytest.mark.parametrize("scale", [1.0, 2.5, 0.01])
def test_scale_other_than_inverse_sqrt_d(ga, scale):
    """The backward carries the softmax scale on P (its exponent is shifted by
    ln(scale)); scales at and above 1 and far below 1/sqrt(d) exercise both
    signs of that shift."""
    b, s, hq, hkv, d, window, seed = 1, 300, 4, 2, 128, 90, 21
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=seed, with_dout=True)
    if scale >= 1:  # keep the scores in the range a trained model produces
        q, k = (q.float() * 0.3).to(torch.bfloat16), (k.float() * 0.3).to(torch.bfloat16)
    ids, pos = workload.random_segments(b, s, seed=seed)
    x = dict(q=q, k=k, v=v, dout=dout, ids=ids, pos=pos)
    _full_check(ga, x, window, scale)

def _sampled(ga, name, dq_samples, key_samples, det=False):
    w = workload.WORKLOADS[name]
    x = workload.make(w, device=DEV, with_dout=True)
    out, lse = ga.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], window_left=w.window_left,
                           scale=w.scale)
    dq, dk, dv = ga.attn_bwd(x["q"], x["k"], x["v"], out, lse, x["dout"], x["ids"], x["pos"],
                             window_left=w.window_left, scale=w.scale, deterministic=det,
                             check_status=True)
    torch.cuda.synchronize()
    del out, lse
    ids, pos = x["ids"].cpu(), x["pos"].cpu()
    g = w.hq // w.hkv
    for bi, kvh, r0, nrows in dq_samples:
        rows = np.arange(r0, r0 + nrows)
        hs = slice(kvh * g, kvh * g + g)
        sl = dict(q=x["q"][bi:bi + 1, :, hs].cpu(), k=x["k"][bi:bi + 1, :, kvh:kvh + 1].cpu(),
                  v=x["v"][bi:bi + 1, :, kvh:kvh + 1].cpu(),
                  dout=x["dout"][bi:bi + 1, :, hs].cpu())
        rq, _, _ = A.attn_bwd(sl["q"], sl["k"], sl["v"], sl["dout"], ids[bi:bi + 1],
                              pos[bi:bi + 1], ids[bi:bi + 1], pos[bi:bi + 1], w.window_left,
                              w.scale, rows=rows)
        check_grad(dq[bi, r0:r0 + nrows, hs].cpu(), rq[0, rows], f"dq b{bi} kvh{kvh} r{r0}")
    for bi, kvh, k0, nkeys in key_samples:
        keys = np.arange(k0, k0 + nkeys)
        rows = A.rows_seeing_keys(ids[bi], pos[bi], ids[bi], pos[bi], w.window_left, keys)
        hs = slice(kvh * g, kvh * g + g)
        sl = dict(q=x["q"][bi:bi + 1, :, hs].cpu(), k=x["k"][bi:bi + 1, :, kvh:kvh + 1].cpu(),
                  v=x["v"][bi:bi + 1, :, kvh:kvh + 1].cpu(),
                  dout=x["dout"][bi:bi + 1, :, hs].cpu())
        _, rk, rv = A.attn_bwd(sl["q"], sl["k"], sl["v"], sl["dout"], ids[bi:bi + 1],
                               pos[bi:bi + 1], ids[bi:bi + 1], pos[bi:bi + 1], w.window_left,
                               w.scale, rows=rows)
        check_grad(dk[bi, k0:k0 + nkeys, kvh].cpu(), rk[0, keys, 0], f"dk b{bi} kvh{kvh} k{k0}")
        check_grad(dv[bi, k0:k0 + nkeys, kvh].cpu(), rv[0, keys, 0], f"dv b{bi} kvh{kvh} k{k0}")
    pad = (ids == 0).to(DEV)
    assert torch.all(dq[pad] == 0) and torch.all(dk[pad] == 0) and torch.all(dv[pad] == 0)
    del x, dq, dk, dv
    torch.cuda.empty_cache()


def test_packed_swa_sampled(ga):
    _sampled(ga, "packed_swa",
             dq_samples=[(0, 0, 0, 128), (1, 7, 4096 + 2000, 200), (0, 3, 3 * 4096 + 2900, 200)],
             key_samples=[(0, 2, 1900, 128), (1, 5, 4096 + 3000, 72), (0, 0, 0, 64)])


@pytest.mark.parametrize("det", [False, True])
def test_full_swa_64k_sampled(ga, det):
    """The 64k packed GQA-SWA workload in the benchmark's launch configuration
    (and in deterministic mode)."""
    _sampled(ga, "full_swa_64k",
             dq_samples=[(0, 0, 9000, 64), (1, 7, 16384 + 12200, 120)],
             key_samples=[(0, 3, 12160, 128), (1, 6, 2 * 16384 + 12220, 68)], det=det)


def test_packed_kv_layout_fwd_bwd():
    """THD_T2HD (TE tutorial section 1): k and v interleaved in one
    [b, s, 2, h_kv, d] tensor, passed as strided views; dk / dv come back in
    the same packed layout.  Same results as the oracle on contiguous k, v."""
    import long_context_attention_attn_gb300 as ga
    from oracle import attention as A
    b, s, hq, hkv, d, window = 2, 1000, 4, 2, 128, 300
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=31, with_dout=True)
    ids, pos = workload.segments(b, s, None)
    kv = torch.stack([k, v], dim=2).cuda()          # [b, s, 2, hkv, d]
    kd, vd = kv[:, :, 0], kv[:, :, 1]
    assert not kd.is_contiguous()
    qd, idd, pd, dod = q.cuda(), ids.cuda(), pos.cuda(), dout.cuda()
    out, lse = ga.attn_fwd(qd, kd, vd, idd, pd, window_left=window, scale=d ** -0.5)
    dq, dk, dv = ga.attn_bwd(qd, kd, vd, out, lse, dod, idd, pd, window_left=window,
                             scale=d ** -0.5)
    torch.cuda.synchronize()
    assert dk.stride() == kd.stride() and dv.data_ptr() - dk.data_ptr() == hkv * d * 2
    ro, rl = A.attn_fwd(q, k, v, ids, pos, ids, pos, window, d ** -0.5)
    check_out(out.cpu(), ro)
    check_lse(lse.cpu(), rl)
    gq, gk, gv = A.attn_bwd(q, k, v, dout, ids, pos, ids, pos, window, d ** -0.5)
    check_grad(dq.cpu(), gq, "dq")
    check_grad(dk.cpu(), gk, "dk")
    check_grad(dv.cpu(), gv, "dv")


def test_full_swa_64k_whole_slot_of_one_group(ga):
    """The 64k workload in the benchmark's launch configuration, checked on one
    whole slot (batch row 1, tokens 16384-32767: segment 2 and its padding) of
    one kv group (kv head 5, query heads 80-95): every element of out, lse, dQ,
    dK and dV there.  Segments see only themselves, so the oracle run on the
    slot's tokens alone gives exactly these rows, and dK / dV of the slot's keys
    are complete (every query row that sees them is in the slot)."""
    import os
    w = workload.WORKLOADS["full_swa_64k"]
    x = workload.make(w, device=DEV, with_dout=True)
    out, lse = ga.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], window_left=w.window_left,
                           scale=w.scale)
    dq, dk, dv = ga.attn_bwd(x["q"], x["k"], x["v"], out, lse, x["dout"], x["ids"], x["pos"],
                             window_left=w.window_left, scale=w.scale)
    torch.cuda.synchronize()
    bi, kvh, t0, t1 = 1, 5, 16384, 32768
    g = w.hq // w.hkv
    hs = slice(kvh * g, kvh * g + g)
    cut = lambda t, h: t[bi:bi + 1, t0:t1, h].cpu()
    q, k, v, do = cut(x["q"], hs), cut(x["k"], slice(kvh, kvh + 1)), \
        cut(x["v"], slice(kvh, kvh + 1)), cut(x["dout"], hs)
    ids, pos = x["ids"][bi:bi + 1, t0:t1].cpu(), x["pos"][bi:bi + 1, t0:t1].cpu()
    got = dict(out=cut(out, hs), lse=lse[bi:bi + 1, hs, t0:t1].cpu(), dq=cut(dq, hs),
               dk=cut(dk, slice(kvh, kvh + 1)), dv=cut(dv, slice(kvh, kvh + 1)))
    del x, out, lse, dq, dk, dv
    torch.cuda.empty_cache()
    torch.set_num_threads(os.cpu_count() or 1)
    ro, rl = A.attn_fwd(q, k, v, ids, pos, ids, pos, w.window_left, w.scale)
    check_out(got["out"], ro)
    check_lse(got["lse"], rl)
    rq, rk, rv = A.attn_bwd(q, k, v, do, ids, pos, ids, pos, w.window_left, w.scale, out=ro)
    check_grad(got["dq"], rq, "dq")
    check_grad(got["dk"], rk, "dk")
    check_grad(got["dv"], rv, "dv")
    pad = ids[0] == 0
    assert torch.all(got["out"][0, pad] == 0) and torch.all(got["dq"][0, pad] == 0)
    assert torch.all(got["dk"][0, pad] == 0) and torch.all(got["dv"][0, pad] == 0)


@pytest.mark.parametrize("det", [False, True])
def test_delta_output_is_rowsum_of_dout_times_out(det):
    """attn_bwd's optional D output: rowsum(dO * O) of every query row and
    head (fp64 reference from the same bf16 tensors), summing to vdot(out,
    dout); passing it changes no gradient."""
    import long_context_attention_attn_gb300 as ga
    w = workload.WORKLOADS["packed_swa"]
    x = workload.make(w, device=DEV, with_dout=True)
    q, k, v, ids, pos, dout = x["q"], x["k"], x["v"], x["ids"], x["pos"], x["dout"]
    kw = dict(window_left=w.window_left, scale=w.scale, deterministic=det)
    out, lse = ga.attn_fwd(q, k, v, ids, pos, window_left=w.window_left, scale=w.scale)
    ref = ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, **kw)
    delta = torch.full((w.b, w.hq, w.s), float("nan"), dtype=torch.float32, device=DEV)
    got = ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, delta=delta, check_status=True, **kw)
    torch.cuda.synchronize()
    want = (dout.double() * out.double()).sum(-1).permute(0, 2, 1)  # [b, Hq, s]
    assert torch.allclose(delta.double(), want, rtol=1e-5, atol=1e-5)
    loss = (dout.double() * out.double()).sum()
    assert abs(delta.double().sum().item() - loss.item()) <= 1e-6 * max(1.0, abs(loss.item())) + 1e-2
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    if det:
        assert torch.equal(got[0], ref[0])


@pytest.mark.parametrize("det", [False, True])
def test_stale_workspace_changes_no_result(det):
    """The workspace is scratch: filled with NaN bytes before the call, it
    changes no result.  (The fp32 dQ accumulator rows of query tiles that
    see no key are neither cleared by the pre-pass nor read by the finalise;
    their dq is written as zeros.)"""
    import long_context_attention_attn_gb300 as ga
    w = workload.WORKLOADS["packed_swa"]
    x = workload.make(w, device=DEV, with_dout=True)
    q, k, v, ids, pos, dout = x["q"], x["k"], x["v"], x["ids"], x["pos"], x["dout"]
    kw = dict(window_left=w.window_left, scale=w.scale, deterministic=det)
    out, lse = ga.attn_fwd(q, k, v, ids, pos, window_left=w.window_left, scale=w.scale)
    ref = ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, **kw)
    need = ga.workspace_bytes_bwd(q, k, ids, pos, w.window_left, v=v, deterministic=det)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)  # fp32 NaN everywhere
    got = ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, workspace=ws, check_status=True, **kw)
    torch.cuda.synchronize()
    for g in got:
        assert torch.isfinite(g).all()
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    if det:
        assert torch.equal(got[0], ref[0])
    else:  # dQ sums with unordered fp32 reduce-adds
        check_grad(got[0].cpu(), ref[0].cpu(), "dq")
    pad = ids == 0
    assert torch.all(got[0][pad] == 0)


def test_stale_forward_workspace_changes_no_result():
    """attn_fwd's workspace (tile plan, work order) filled with NaN bytes
    before the call: out and lse bit-identical to a call on a fresh one."""
    import long_context_attention_attn_gb300 as ga
    w = workload.WORKLOADS["packed_swa"]
    x = workload.make(w, device=DEV, with_dout=False)
    q, k, v, ids, pos = x["q"], x["k"], x["v"], x["ids"], x["pos"]
    out, lse = ga.attn_fwd(q, k, v, ids, pos, window_left=w.window_left, scale=w.scale)
    need = ga.workspace_bytes_fwd(q, k, ids, pos, window_left=w.window_left, v=v)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)
    out2, lse2 = ga.attn_fwd(q, k, v, ids, pos, window_left=w.window_left, scale=w.scale,
                             workspace=ws, check_status=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
