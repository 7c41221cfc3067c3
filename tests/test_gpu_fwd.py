"""GPU parity of attn_fwd through the C ABI against the CPU oracle.

Small cases are checked on every element; the large workloads on sampled
(batch, head, row-block) outputs that the oracle computes row by row, in the
same launch configuration the benchmark times."""
import numpy as np
import pytest
import torch

import workload
from oracle import attention as A
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ga():
    import long_context_attention_attn_gb300 as pkg
    return pkg


def _run(ga, q, k, v, ids, pos, kv_ids, kv_pos, window, scale, out_fp32=False):
    out, lse = ga.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), ids.to(DEV), pos.to(DEV),
                           kv_ids.to(DEV), kv_pos.to(DEV), window_left=window, scale=scale,
                           out_fp32=out_fp32)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def _full_check(ga, q, k, v, ids, pos, window, scale, kv_ids=None, kv_pos=None, out_fp32=False):
    kv_ids = ids if kv_ids is None else kv_ids
    kv_pos = pos if kv_pos is None else kv_pos
    out, lse = _run(ga, q, k, v, ids, pos, kv_ids, kv_pos, window, scale, out_fp32)
    ro, rl = A.attn_fwd(q, k, v, ids, pos, kv_ids, kv_pos, window, scale)
    check_out(out, ro)
    check_lse(lse, rl)
    # rows with no visible key are exactly zero
    empty = np.isneginf(rl)  # [b, h, s]
    o = out.float().numpy()
    for bi, h, i in np.argwhere(empty):
        assert np.all(o[bi, i, h] == 0.0)
    return out, lse


def test_tiny_workload(ga):
    w = workload.WORKLOADS["tiny"]
    x = workload.make(w)
    _full_check(ga, x["q"], x["k"], x["v"], x["ids"], x["pos"], w.window_left, w.scale)


@pytest.mark.parametrize("b,s,hq,hkv,d,window,seed", [
    (2, 300, 4, 1, 128, 70, 1),     # ragged tail, g = 4
    (1, 200, 3, 1, 64, -1, 2),      # odd group size: the last pair has one head
    (1, 384, 2, 2, 128, -1, 3),     # g = 1 (plain MHA)
    (2, 517, 8, 2, 64, 0, 4),       # window 0: each token sees only itself
    (1, 1024, 2, 1, 128, 300, 5),
    (2, 300, 4, 2, 256, 70, 6),     # d = 256 (one head per CTA), ragged tail
    (1, 520, 3, 1, 256, -1, 7),     # d = 256, odd group size
    (1, 1000, 2, 2, 256, 0, 8),     # d = 256, window 0
    (2, 6000, 2, 1, 128, 700, 9),   # plan above 4096 class bytes: the parallel plan kernels
])
def test_random_packing(ga, b, s, hq, hkv, d, window, seed):
    q, k, v = workload.qkv(b, s, hq, hkv, d, seed=seed)
    ids, pos = workload.random_segments(b, s, seed=seed)
    _full_check(ga, q, k, v, ids, pos, window, d ** -0.5)


@pytest.mark.parametrize("d", [128, 256])
def test_fp32_output(ga, d):
    q, k, v = workload.qkv(1, 256, 2, 1, d, seed=9)
    ids, pos = workload.segments(1, 256, 2)
    _full_check(ga, q, k, v, ids, pos, -1, 0.1, out_fp32=True)


@pytest.mark.parametrize("b,s,hq,hkv,window,slots,seed", [
    (2, 300, 4, 2, 70, None, 12),    # ragged tail, window
    (1, 520, 3, 1, -1, None, 13),    # odd group size
    (2, 1024, 8, 2, 200, 4, 14),     # padded slots (the tutorial's packing)
])
def test_mla_head_dims(ga, b, s, hq, hkv, window, slots, seed):
    """d_qk = 192, d_v = 128 (MLA): out has V's head dim."""
    q, k, v = workload.qkv(b, s, hq, hkv, 192, seed=seed, dv=128)
    if slots is None:
        ids, pos = workload.random_segments(b, s, seed=seed)
    else:
        ids, pos = workload.segments(b, s, slots)
    out, _ = _full_check(ga, q, k, v, ids, pos, window, 192 ** -0.5)
    assert out.shape == (b, s, hq, 128)


def test_mla_fp32_output(ga):
    q, k, v = workload.qkv(1, 256, 2, 1, 192, seed=15, dv=128)
    ids, pos = workload.segments(1, 256, 2)
    _full_check(ga, q, k, v, ids, pos, -1, 0.1, out_fp32=True)


def test_unsupported_head_dim_is_rejected_before_launch(ga):
    """A head dim outside {64, 128, 256, (192, 128)} fails loudly before any
    launch, in the forward and in the backward."""
    q, k, v, dout = workload.qkv(1, 256, 2, 1, 96, seed=10, with_dout=True)
    ids, pos = workload.segments(1, 256, 1)
    g = {n: t.to(DEV) for n, t in dict(q=q, k=k, v=v, dout=dout, ids=ids, pos=pos).items()}
    with pytest.raises(RuntimeError):
        ga.attn_fwd(g["q"], g["k"], g["v"], g["ids"], g["pos"], scale=96 ** -0.5)
    out = torch.zeros_like(g["q"])
    lse = torch.zeros(1, 2, 256, device=DEV)
    with pytest.raises(RuntimeError):
        ga.attn_bwd(g["q"], g["k"], g["v"], out, lse, g["dout"], g["ids"], g["pos"],
                    scale=96 ** -0.5)


def test_cross_descriptor_and_lengths(ga):
    """Queries of one shard against keys of another (different lengths)."""
    q, _, _ = workload.qkv(1, 256, 4, 2, 128, seed=11)
    _, k, v = workload.qkv(1, 384, 4, 2, 128, seed=12)
    ids = torch.ones(1, 256, dtype=torch.int32)
    pos = torch.arange(300, 556, dtype=torch.int32)[None]
    kv_ids = torch.ones(1, 384, dtype=torch.int32)
    kv_pos = torch.arange(0, 384, dtype=torch.int32)[None]
    kv_ids[0, 100:130] = 0
    _full_check(ga, q, k, v, ids, pos, 200, 0.088, kv_ids, kv_pos)


def test_all_padding_and_single_token(ga):
    q, k, v = workload.qkv(1, 130, 2, 1, 64, seed=13)
    ids = torch.zeros(1, 130, dtype=torch.int32)
    pos = torch.zeros(1, 130, dtype=torch.int32)
    ids[0, 129] = 5
    _full_check(ga, q, k, v, ids, pos, -1, 0.125)


def test_extreme_scores(ga):
    """Large score ranges exercise the stale-max rescaling."""
    q, k, v = workload.qkv(1, 512, 2, 1, 128, seed=14)
    q = (q.float() * 6).to(torch.bfloat16)
    ids, pos = workload.segments(1, 512, None)
    _full_check(ga, q, k, v, ids, pos, -1, 0.3)


def test_packed_thd_workload_all_heads(ga):
    """The packed THD workload on every element: both batch rows, all 16 query
    heads of both kv groups, valid and padding rows."""
    w = workload.WORKLOADS["packed_thd"]
    x = workload.make(w)
    out, lse = _run(ga, x["q"], x["k"], x["v"], x["ids"], x["pos"], x["ids"], x["pos"],
                    w.window_left, w.scale)
    ro, rl = A.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], x["ids"], x["pos"],
                        w.window_left, w.scale)
    check_out(out, ro)
    check_lse(lse, rl)
    pad = (x["ids"] == 0)
    assert torch.all(out[pad] == 0)
    assert torch.all(torch.isneginf(lse.permute(0, 2, 1)[pad]))


def _sampled_check(ga, name, samples):
    w = workload.WORKLOADS[name]
    x = workload.make(w, device=DEV, with_dout=False)
    out, lse = ga.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"],
                           window_left=w.window_left, scale=w.scale)
    torch.cuda.synchronize()
    ids, pos = x["ids"].cpu(), x["pos"].cpu()
    for bi, h, r0, nrows in samples:
        rows = np.arange(r0, r0 + nrows)
        kvh = h // (w.hq // w.hkv)
        q1 = x["q"][bi:bi + 1, :, h:h + 1].cpu()
        k1 = x["k"][bi:bi + 1, :, kvh:kvh + 1].cpu()
        v1 = x["v"][bi:bi + 1, :, kvh:kvh + 1].cpu()
        ro, rl = A.attn_fwd(q1, k1, v1, ids[bi:bi + 1], pos[bi:bi + 1], ids[bi:bi + 1],
                            pos[bi:bi + 1], w.window_left, w.scale, rows=rows)
        check_out(out[bi, r0:r0 + nrows, h].cpu(), ro[0, rows, 0], f"out b{bi} h{h} r{r0}")
        check_lse(lse[bi, h, r0:r0 + nrows].cpu(), rl[0, 0, rows], f"lse b{bi} h{h} r{r0}")
    del x, out, lse
    torch.cuda.empty_cache()


def test_packed_swa_sampled(ga):
    _sampled_check(ga, "packed_swa", [(0, 0, 0, 128), (1, 31, 3000, 200), (0, 9, 4096 + 2900, 300),
                                      (1, 17, 16384 - 200, 200)])


def test_ring_workload_full_attention_sampled(ga):
    _sampled_check(ga, "ring_cp4", [(0, 0, 0, 128), (0, 63, 32768 - 128, 128), (0, 20, 15000, 64)])


def test_full_swa_64k_sampled(ga):
    """The 64k packed GQA-SWA workload, in the benchmark's launch configuration."""
    _sampled_check(ga, "full_swa_64k", [
        (0, 0, 0, 128),                  # slot start
        (0, 127, 12288 - 128, 160),      # end of slot 1 valid part + padding rows
        (1, 64, 16384 + 9000, 128),      # window fully active
        (1, 1, 3 * 16384 + 8100, 200),   # window edge crossing
    ])


@pytest.mark.parametrize("name,samples", [
    ("packed_swa_d256", [(0, 0, 0, 128), (1, 31, 4096 + 2900, 300), (0, 12, 16384 - 200, 200)]),
    ("packed_swa_mla", [(0, 3, 1000, 128), (1, 30, 2 * 4096 + 3000, 200)]),
    ("causal_32k_d256", [(0, 0, 0, 128), (0, 31, 32768 - 100, 100), (0, 9, 20000, 64)]),
    ("causal_32k_mla", [(0, 5, 127, 130), (0, 26, 32768 - 64, 64)]),
])
def test_other_head_dims_sampled(ga, name, samples):
    """The forward-only head-dim workloads at the sizes the bench times them."""
    _sampled_check(ga, name, samples)


def test_fwd_bit_identical_across_repeats(ga):
    """The forward has a fixed reduction order, so repeated calls must agree bit
    for bit; a read of O before the last P.V groups land (or any other race
    between the MMA and softmax warps) shows up as run-to-run differences.
    A short window gives every query tile only a few key tiles, so each of
    the launch's many CTAs reaches its epilogue while its last P.V groups are
    still close behind — the case that exposed such a race."""
    b, s, hq, hkv, d = 2, 8192, 16, 2, 128
    q, k, v = (t.cuda() for t in workload.qkv(b, s, hq, hkv, d, seed=99))
    ids, pos = (t.cuda() for t in workload.segments(b, s, None))
    first = None
    for _ in range(12):
        o, l = ga.attn_fwd(q, k, v, ids, pos, window_left=100, scale=d ** -0.5)
        torch.cuda.synchronize()
        if first is None:
            first = (o.clone(), l.clone())
        else:
            assert torch.equal(o, first[0]) and torch.equal(l, first[1])
