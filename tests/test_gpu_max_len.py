"""GPU parity at the largest sequence the work order is built for: one batch
row of 2^20 tokens (one causal segment with a 100-token padding tail, window
(2047, 0), Hq 8, Hkv 2, d 128), forward and backward through the C ABI.

The CPU oracle sees only local slices: a query row with window w sees keys
no further back than w positions, so the oracle run on tokens [r0 - w, r1)
(with their original segment ids and positions) gives exactly the rows
[r0, r1); the keys [k0, k1) are seen only by rows up to k1 - 1 + w, so the
slice [k0 - w, k1 + w) holds every contribution to their dK / dV."""
import numpy as np
import pytest
import torch

import workload
from oracle import attention as A
from tests.parity import check_grad, check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"
S, HQ, HKV, D, WINDOW, PAD = 1 << 20, 8, 2, 128, 2047, 100
VALID = S - PAD


@pytest.fixture(scope="module")
def ga():
    import long_context_attention_attn_gb300 as pkg
    return pkg


@pytest.fixture(scope="module")
def inputs():
    q, k, v, dout = workload.qkv(1, S, HQ, HKV, D, seed=97, with_dout=True, device=DEV)
    ids = torch.ones(1, S, dtype=torch.int32)
    ids[0, VALID:] = 0
    pos = torch.arange(S, dtype=torch.int32)[None].clone()
    pos[0, VALID:] = 0
    return dict(q=q, k=k, v=v, dout=dout, ids=ids.to(DEV), pos=pos.to(DEV),
                ids_cpu=ids, pos_cpu=pos)


def _slice(x, a, e):
    cut = lambda t: t[:, a:e].cpu()
    return (cut(x["q"]), cut(x["k"]), cut(x["v"]), cut(x["dout"]),
            x["ids_cpu"][:, a:e], x["pos_cpu"][:, a:e])


# query rows: the first tile, a run across tile boundaries in the middle,
# the last valid rows (the ragged tail of the last tile)
DQ_ROWS = [(0, 128), ((1 << 19) + 1000, 200), (VALID - 200, 200)]
# key blocks: the first keys, a run straddling a tile boundary, the last valid keys
KEY_BLOCKS = [(0, 64), ((1 << 19) - 40, 100), (VALID - 72, 72)]


def _check_rows(x, out, lse, dq):
    for r0, n in DQ_ROWS:
        a = max(0, r0 - WINDOW)
        q, k, v, do, ids, pos = _slice(x, a, r0 + n)
        rows = np.arange(r0 - a, r0 - a + n)
        ro, rl = A.attn_fwd(q, k, v, ids, pos, ids, pos, WINDOW, D ** -0.5, rows=rows)
        check_out(out[0, r0:r0 + n].cpu(), ro[0, rows], f"out r{r0}")
        check_lse(lse[0, :, r0:r0 + n].cpu(), rl[0][:, rows], f"lse r{r0}")
        rq, _, _ = A.attn_bwd(q, k, v, do, ids, pos, ids, pos, WINDOW, D ** -0.5, rows=rows)
        check_grad(dq[0, r0:r0 + n].cpu(), rq[0, rows], f"dq r{r0}")


def _check_keys(x, dk, dv):
    for k0, n in KEY_BLOCKS:
        a, e = max(0, k0 - WINDOW), min(S, k0 + n + WINDOW)
        q, k, v, do, ids, pos = _slice(x, a, e)
        keys = np.arange(k0 - a, k0 - a + n)
        rows = A.rows_seeing_keys(ids[0], pos[0], ids[0], pos[0], WINDOW, keys)
        assert rows.size > 0
        _, rk, rv = A.attn_bwd(q, k, v, do, ids, pos, ids, pos, WINDOW, D ** -0.5, rows=rows)
        check_grad(dk[0, k0:k0 + n].cpu(), rk[0, keys], f"dk k{k0}")
        check_grad(dv[0, k0:k0 + n].cpu(), rv[0, keys], f"dv k{k0}")


@pytest.mark.parametrize("det", [False, True])
def test_one_row_of_2_pow_20_tokens(ga, inputs, det):
    x = inputs
    out, lse = ga.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], window_left=WINDOW,
                           scale=D ** -0.5, check_status=True)
    dq, dk, dv = ga.attn_bwd(x["q"], x["k"], x["v"], out, lse, x["dout"], x["ids"], x["pos"],
                             window_left=WINDOW, scale=D ** -0.5, deterministic=det,
                             check_status=True)
    torch.cuda.synchronize()
    _check_rows(x, out, lse, dq)
    _check_keys(x, dk, dv)
    pad = slice(VALID, S)
    assert torch.all(out[0, pad] == 0) and torch.all(dq[0, pad] == 0)
    assert torch.all(dk[0, pad] == 0) and torch.all(dv[0, pad] == 0)
    assert torch.all(torch.isfinite(lse[0, :, :VALID]))
    del out, lse, dq, dk, dv
    torch.cuda.empty_cache()
