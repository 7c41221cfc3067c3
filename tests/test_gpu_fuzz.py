"""Seeded random configurations through the C ABI against the CPU oracle:
sequence lengths around the kernels' 64- and 128-token tile edges, GQA group
sizes 1-5 (odd groups leave a single-head slot), d = 64 / 128, no window /
random windows, random packings with padding runs, and cross-length calls
(queries of one block against keys of another, as a ring step makes).
Forward (O, LSE) and backward (dQ, dK, dV) are both checked; the forward-only
head dims (256, and MLA's 192 / 128) get forward cases of their own."""
import numpy as np
import pytest
import torch

import workload
from oracle import attention as A
from tests.parity import check_grad, check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"

LENGTHS = [1, 2, 63, 64, 65, 127, 128, 129, 191, 255, 257, 383, 640, 1000, 1500]


def _config(seed: int):
    rng = np.random.default_rng(1000 + seed)
    b = int(rng.integers(1, 3))
    s_q = int(rng.choice(LENGTHS))
    cross = bool(rng.random() < 0.3)
    s_kv = int(rng.choice(LENGTHS)) if cross else s_q
    hkv = int(rng.integers(1, 3))
    g = int(rng.integers(1, 6))
    d = int(rng.choice([64, 128]))
    window = -1 if rng.random() < 0.4 else int(rng.integers(0, max(1, s_kv)))
    return b, s_q, s_kv, hkv * g, hkv, d, window, cross


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_fwd_bwd(seed):
    import long_context_attention_attn_gb300 as ga
    b, s_q, s_kv, hq, hkv, d, window, cross = _config(seed)
    q, _, _, dout = workload.qkv(b, s_q, hq, hkv, d, seed=seed, with_dout=True)
    _, k, v = workload.qkv(b, s_kv, hq, hkv, d, seed=seed + 500)
    ids, pos = workload.random_segments(b, s_q, seed=seed, max_segments=3, pad_prob=0.25)
    if cross:
        # keys of an earlier block of the same sequence: one segment, shifted
        # positions, a padding run
        kv_ids = torch.ones(b, s_kv, dtype=torch.int32)
        kv_pos = torch.arange(s_kv, dtype=torch.int32)[None].repeat(b, 1)
        kv_ids[:, s_kv // 3: s_kv // 3 + s_kv // 7] = 0
        ids = torch.ones(b, s_q, dtype=torch.int32)
        pos = torch.arange(s_kv // 2, s_kv // 2 + s_q, dtype=torch.int32)[None].repeat(b, 1)
    else:
        kv_ids, kv_pos = ids, pos
    scale = d ** -0.5
    dv_ = {n: t.to(DEV) for n, t in (("q", q), ("k", k), ("v", v), ("dout", dout), ("ids", ids),
                                       ("pos", pos), ("kv_ids", kv_ids), ("kv_pos", kv_pos))}
    out, lse = ga.attn_fwd(dv_["q"], dv_["k"], dv_["v"], dv_["ids"], dv_["pos"], dv_["kv_ids"],
                           dv_["kv_pos"], window_left=window, scale=scale)
    dq, dk, dvv = ga.attn_bwd(dv_["q"], dv_["k"], dv_["v"], out, lse, dv_["dout"], dv_["ids"],
                              dv_["pos"], dv_["kv_ids"], dv_["kv_pos"], window_left=window,
                              scale=scale)
    torch.cuda.synchronize()
    ro, rl = A.attn_fwd(q, k, v, ids, pos, kv_ids, kv_pos, window, scale)
    check_out(out.cpu(), ro)
    check_lse(lse.cpu(), rl)
    rq, rk, rv = A.attn_bwd(q, k, v, dout, ids, pos, kv_ids, kv_pos, window, scale)
    check_grad(dq.cpu(), rq, "dq")
    check_grad(dk.cpu(), rk, "dk")
    check_grad(dvv.cpu(), rv, "dv")


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_fwd_wide_heads(seed):
    """Forward-only head dims: d = 256, and d_qk = 192 with d_v = 128 (MLA)."""
    import long_context_attention_attn_gb300 as ga
    b, s_q, s_kv, hq, hkv, _, window, cross = _config(100 + seed)
    d, d_v = (256, 256) if seed % 2 == 0 else (192, 128)
    q, _, _ = workload.qkv(b, s_q, hq, hkv, d, seed=seed)
    _, k, v = workload.qkv(b, s_kv, hq, hkv, d, seed=seed + 500, dv=d_v)
    ids, pos = workload.random_segments(b, s_q, seed=seed, max_segments=3, pad_prob=0.25)
    if cross:
        kv_ids = torch.ones(b, s_kv, dtype=torch.int32)
        kv_pos = torch.arange(s_kv, dtype=torch.int32)[None].repeat(b, 1)
        ids = torch.ones(b, s_q, dtype=torch.int32)
        pos = torch.arange(s_kv // 2, s_kv // 2 + s_q, dtype=torch.int32)[None].repeat(b, 1)
    else:
        kv_ids, kv_pos = ids, pos
    scale = d ** -0.5
    g = {n: t.to(DEV) for n, t in (("q", q), ("k", k), ("v", v), ("ids", ids), ("pos", pos),
                                   ("kv_ids", kv_ids), ("kv_pos", kv_pos))}
    out, lse = ga.attn_fwd(g["q"], g["k"], g["v"], g["ids"], g["pos"], g["kv_ids"], g["kv_pos"],
                           window_left=window, scale=scale)
    torch.cuda.synchronize()
    assert out.shape == (b, s_q, hq, d_v)
    ro, rl = A.attn_fwd(q, k, v, ids, pos, kv_ids, kv_pos, window, scale)
    check_out(out.cpu(), ro)
    check_lse(lse.cpu(), rl)
