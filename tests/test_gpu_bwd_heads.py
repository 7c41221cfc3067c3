"""GPU parity of attn_bwd at the head dims the dK / dV + dQ kernel pair serves:
d = 256, and the MLA shape d_qk = 192 with d_v = 128 (TE tutorial, "Next
steps").  Every element of dQ, dK and dV is compared with the CPU oracle
(explicit-P float64 backward) on small and irregular cases, including
lengths around the 64 / 128 tile edges, GQA groups 1-5, windows, separate
query / key descriptors, the fp32 accumulate mode the ring backward uses, and
sampled rows / key tiles at the packed_swa packing."""
import numpy as np
import pytest
import torch

import workload
from oracle import attention as A
from tests.parity import check_grad, check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"
HEADS = [(256, 256), (192, 128)]


@pytest.fixture(scope="module")
def ga():
    import long_context_attention_attn_gb300 as pkg
    return pkg


def _fwd_bwd(ga, x, window, scale, kv=None):
    g = {k: v.to(DEV) for k, v in x.items()}
    kv_ids = g.get("kv_ids", g["ids"])
    kv_pos = g.get("kv_pos", g["pos"])
    out, lse = ga.attn_fwd(g["q"], g["k"], g["v"], g["ids"], g["pos"], kv_ids, kv_pos,
                           window_left=window, scale=scale, check_status=True)
    dq, dk, dv = ga.attn_bwd(g["q"], g["k"], g["v"], out, lse, g["dout"], g["ids"], g["pos"],
                             kv_ids, kv_pos, window_left=window, scale=scale, check_status=True)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()


def _check_all(ga, x, window, scale):
    kv_ids = x.get("kv_ids", x["ids"])
    kv_pos = x.get("kv_pos", x["pos"])
    out, lse, dq, dk, dv = _fwd_bwd(ga, x, window, scale)
    ro, rl = A.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], kv_ids, kv_pos, window, scale)
    check_out(out, ro)
    check_lse(lse, rl)
    rq, rk, rv = A.attn_bwd(x["q"], x["k"], x["v"], x["dout"], x["ids"], x["pos"], kv_ids, kv_pos,
                            window, scale, out=ro)
    check_grad(dq, rq, "dq")
    check_grad(dk, rk, "dk")
    check_grad(dv, rv, "dv")
    # rows that see no key and keys no row sees get exactly zero gradients
    blind = torch.from_numpy(np.abs(ro).sum(axis=(2, 3)) == 0)
    assert torch.all(dq[blind] == 0)
    unseen = torch.from_numpy((np.abs(rk).sum(axis=(2, 3)) == 0) & (np.abs(rv).sum(axis=(2, 3)) == 0))
    assert torch.all(dk[unseen] == 0) and torch.all(dv[unseen] == 0)


def _inputs(b, s, hq, hkv, d, dv, seed, packing="random"):
    q, k, v, dout = workload.qkv(b, s, hq, hkv, d, seed=seed, with_dout=True, dv=dv)
    if packing == "random":
        ids, pos = workload.random_segments(b, s, seed=seed)
    else:
        ids, pos = workload.segments(b, s, packing)
    return dict(q=q, k=k, v=v, dout=dout, ids=ids, pos=pos)


@pytest.mark.parametrize("d,dv", HEADS)
@pytest.mark.parametrize("b,s,hq,hkv,window,seed", [
    (2, 300, 4, 1, 70, 1),     # ragged tail, g = 4
    (1, 200, 3, 1, -1, 2),     # odd group
    (1, 384, 2, 2, -1, 3),     # g = 1, whole tiles
    (1, 640, 4, 2, 0, 4),      # window 0 (each row sees itself)
    (1, 129, 5, 1, 40, 5),     # one row past a tile, g = 5
    (2, 63, 2, 1, -1, 6),      # shorter than a 64-row step
])
def test_random_packing(ga, d, dv, b, s, hq, hkv, window, seed):
    _check_all(ga, _inputs(b, s, hq, hkv, d, dv, seed), window, d ** -0.5)


@pytest.mark.parametrize("d,dv", HEADS)
def test_padded_slots_and_tiny_workload_shape(ga, d, dv):
    """The tutorial's padded-slot packing (ids 1..4, 0 on padding) and the
    tiny workload's one-segment causal shape at these head dims."""
    _check_all(ga, _inputs(1, 1024, 4, 2, d, dv, 7, packing=4), 300, d ** -0.5)
    _check_all(ga, _inputs(1, 256, 4, 2, d, dv, 8, packing=None), -1, d ** -0.5)


@pytest.mark.parametrize("d,dv", HEADS)
@pytest.mark.parametrize("s_q,s_kv,q0,window,seed", [
    (256, 384, 300, 200, 11),   # queries late in the key range
    (200, 520, 100, -1, 12),    # ragged on both sides
    (384, 130, 0, 40, 13),      # more queries than keys
])
def test_cross_descriptor_and_lengths(ga, d, dv, s_q, s_kv, q0, window, seed):
    """Queries of one shard against keys of another (a ring step's call),
    with a padding hole in the keys."""
    hq, hkv = 4, 2
    q, _, _, dout = workload.qkv(1, s_q, hq, hkv, d, seed=seed, with_dout=True, dv=dv)
    _, k, v = workload.qkv(1, s_kv, hq, hkv, d, seed=seed + 100, dv=dv)
    ids = torch.ones(1, s_q, dtype=torch.int32)
    pos = torch.arange(q0, q0 + s_q, dtype=torch.int32)[None]
    kv_ids = torch.ones(1, s_kv, dtype=torch.int32)
    kv_pos = torch.arange(0, s_kv, dtype=torch.int32)[None]
    kv_ids[0, s_kv // 3:s_kv // 3 + 30] = 0
    x = dict(q=q, k=k, v=v, dout=dout, ids=ids, pos=pos, kv_ids=kv_ids, kv_pos=kv_pos)
    _check_all(ga, x, window, d ** -0.5)


@pytest.mark.parametrize("d,dv", HEADS)
@pytest.mark.parametrize("scale", [1.0, 0.01])
def test_other_scales(ga, d, dv, scale):
    x = _inputs(1, 300, 4, 2, d, dv, 21)
    if scale >= 1:  # keep the scores in a trained model's range
        x["q"] = (x["q"].float() * 0.2).to(torch.bfloat16)
        x["k"] = (x["k"].float() * 0.2).to(torch.bfloat16)
    _check_all(ga, x, 90, scale)


@pytest.mark.parametrize("d,dv", HEADS)
def test_accumulate_mode_adds(ga, d, dv):
    """accumulate_fp32 (the ring backward's per-block calls): this call's
    gradients are added to the fp32 accumulators' contents."""
    x = _inputs(1, 300, 4, 2, d, dv, 31)
    g = {k: t.to(DEV) for k, t in x.items()}
    out, lse = ga.attn_fwd(g["q"], g["k"], g["v"], g["ids"], g["pos"], window_left=100,
                           scale=d ** -0.5)
    gen = torch.Generator(device=DEV).manual_seed(3)
    base = [torch.randn(t.shape, generator=gen, device=DEV) for t in (g["q"], g["k"], g["v"])]
    acc = [t.clone() for t in base]
    ga.attn_bwd(g["q"], g["k"], g["v"], out, lse, g["dout"], g["ids"], g["pos"],
                window_left=100, scale=d ** -0.5, dq=acc[0], dk=acc[1], dv=acc[2],
                accumulate_fp32=True, check_status=True)
    torch.cuda.synchronize()
    rq, rk, rv = A.attn_bwd(x["q"], x["k"], x["v"], x["dout"], x["ids"], x["pos"], x["ids"],
                            x["pos"], 100, d ** -0.5, out=out.float().cpu())
    for name, a_, b_, ref in (("dq", acc[0], base[0], rq), ("dk", acc[1], base[1], rk),
                              ("dv", acc[2], base[2], rv)):
        check_grad((a_ - b_).cpu(), ref, name)


@pytest.mark.parametrize("d,dv", HEADS)
@pytest.mark.parametrize("seed", range(6))
def test_fuzz_tile_edges(ga, d, dv, seed):
    """Seeded random shapes around the 64 / 128 tile edges, GQA groups 1-5,
    random windows and packings."""
    rng = np.random.default_rng(1000 + seed)
    s = int(rng.choice([63, 64, 65, 127, 128, 129, 191, 255, 257, 400]))
    hkv = int(rng.integers(1, 3))
    hq = hkv * int(rng.integers(1, 6))
    window = int(rng.choice([-1, 0, 17, 100]))
    b = int(rng.integers(1, 3))
    _check_all(ga, _inputs(b, s, hq, hkv, d, dv, 500 + seed), window, d ** -0.5)


@pytest.mark.parametrize("name", ["packed_swa_d256", "packed_swa_mla"])
def test_packed_swa_shapes_sampled(ga, name):
    """The packed_swa packing (b 2, s 16384 in 4 slots of 4096, Hq 32, Hkv 8,
    window 1024) at these head dims, in one full-size launch: dQ on sampled
    query rows, dK / dV on sampled key tiles (complete: every row that sees
    those keys is included), padding exactly zero."""
    w = workload.WORKLOADS[name]
    x = workload.make(w, device=DEV, with_dout=True)
    out, lse = ga.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], window_left=w.window_left,
                           scale=w.scale)
    dq, dk, dv = ga.attn_bwd(x["q"], x["k"], x["v"], out, lse, x["dout"], x["ids"], x["pos"],
                             window_left=w.window_left, scale=w.scale, check_status=True)
    torch.cuda.synchronize()
    ids, pos = x["ids"].cpu(), x["pos"].cpu()
    g = w.hq // w.hkv
    for bi, kvh, r0, nrows in ((0, 0, 0, 128), (1, 7, 4096 + 2000, 200), (0, 3, 3 * 4096 + 2900, 200)):
        rows = np.arange(r0, r0 + nrows)
        hs = slice(kvh * g, kvh * g + g)
        sl = [x[n][bi:bi + 1, :, hs if n in ("q", "dout") else slice(kvh, kvh + 1)].cpu()
              for n in ("q", "k", "v", "dout")]
        rq, _, _ = A.attn_bwd(*sl, ids[bi:bi + 1], pos[bi:bi + 1], ids[bi:bi + 1],
                              pos[bi:bi + 1], w.window_left, w.scale, rows=rows)
        check_grad(dq[bi, r0:r0 + nrows, hs].cpu(), rq[0, rows], f"dq b{bi} kvh{kvh} r{r0}")
    for bi, kvh, k0, nkeys in ((0, 2, 1900, 128), (1, 5, 4096 + 3000, 72)):
        keys = np.arange(k0, k0 + nkeys)
        rows = A.rows_seeing_keys(ids[bi], pos[bi], ids[bi], pos[bi], w.window_left, keys)
        hs = slice(kvh * g, kvh * g + g)
        sl = [x[n][bi:bi + 1, :, hs if n in ("q", "dout") else slice(kvh, kvh + 1)].cpu()
              for n in ("q", "k", "v", "dout")]
        _, rk, rv = A.attn_bwd(*sl, ids[bi:bi + 1], pos[bi:bi + 1], ids[bi:bi + 1],
                               pos[bi:bi + 1], w.window_left, w.scale, rows=rows)
        check_grad(dk[bi, k0:k0 + nkeys, kvh].cpu(), rk[0, keys, 0], f"dk b{bi} kvh{kvh} k{k0}")
        check_grad(dv[bi, k0:k0 + nkeys, kvh].cpu(), rv[0, keys, 0], f"dv b{bi} kvh{kvh} k{k0}")
    pad = (ids == 0).to(DEV)
    assert torch.all(dq[pad] == 0) and torch.all(dk[pad] == 0) and torch.all(dv[pad] == 0)


@pytest.mark.parametrize("d,dv", HEADS)
def test_ring_backward(ga, d, dv):
    """The ring-emulated backward (per-block calls in accumulate mode) at these
    head dims equals the oracle's full backward."""
    from long_context_attention_attn_gb300 import ring
    x = _inputs(1, 2048, 4, 2, d, dv, 41, packing=None)
    g = {k: t.to(DEV) for k, t in x.items()}
    out, lse = ga.attn_fwd(g["q"], g["k"], g["v"], g["ids"], g["pos"], window_left=-1,
                           scale=d ** -0.5)
    dq, dk, dvv = ring.ring_attn_bwd(g["q"], g["k"], g["v"], out, lse, g["dout"], g["ids"],
                                     g["pos"], 4, scale=d ** -0.5)
    torch.cuda.synchronize()
    rq, rk, rv = A.attn_bwd(x["q"], x["k"], x["v"], x["dout"], x["ids"], x["pos"], x["ids"],
                            x["pos"], -1, d ** -0.5)
    check_grad(dq.cpu(), rq, "dq")
    check_grad(dk.cpu(), rk, "dk")
    check_grad(dvv.cpu(), rv, "dv")
