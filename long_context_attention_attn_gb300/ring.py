"""Ring-attention context parallelism emulated on one GPU.

"Context parallelism and ring attention", section "Ring attention": every
shard keeps its query block and, step by step, attends to the key/value block
it currently holds, folding each partial result into a running softmax
(section "Online softmax"), until every block has been seen.  Here the R
shards are logical: the sequence is put in causal load-balancing order
(section "Load balance"; TE tutorial section 4), shard r owns rows
[r*s/R, (r+1)*s/R) of the reordered tensors, and "receiving" block j at step t
(j = (r - t) mod R, the local block first) means reading those rows in place.
Masks use the reordered segment positions, so causality across shard
boundaries follows global positions.

Every step runs in the library's kernels: reorder / inverse reorder,
attn_fwd on shard views (fp32 partial output), attn_merge_partial.  This
module is host control only.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (DUAL_CHUNK, STRIPED, attn_fwd, attn_merge_partial, inverse_reorder_causal_lb,
               reorder_causal_lb, workspace_bytes_fwd)


def ring_attn_fwd(q, k, v, ids, pos, cp_size: int, *, window_left: int = -1,
                  scale: Optional[float] = None, strategy: int = DUAL_CHUNK, stripe_size: int = 1):
    """Forward attention computed as cp_size ring steps per logical shard.

    q bf16 [b,s,Hq,d]; k, v bf16 [b,s,Hkv,d]; ids/pos int32 [b,s] (natural
    order).  Returns (out bf16 [b,s,Hq,d], lse fp32 [b,Hq,s]) in natural order.
    """
    b, s, hq, d = q.shape
    R = int(cp_size)
    if s % R:
        raise ValueError("sequence length must be divisible by cp_size")
    n = s // R
    dev = q.device
    re = lambda x: reorder_causal_lb(x, strategy, R, stripe_size, seq_dim=1)
    qr, kr, vr, idr, posr = re(q), re(k), re(v), re(ids), re(pos)
    out = torch.empty_like(q)
    lse = torch.empty(b, hq, s, dtype=torch.float32, device=dev)
    acc = torch.empty(1, n, hq, d, dtype=torch.float32, device=dev)
    blk = torch.empty(1, n, hq, d, dtype=torch.float32, device=dev)
    blk_lse = torch.empty(1, hq, n, dtype=torch.float32, device=dev)
    lse_sh = torch.empty(R, hq, n, dtype=torch.float32, device=dev)
    out_r = torch.empty(1, s, hq, d, dtype=q.dtype, device=dev)
    ws = torch.empty(workspace_bytes_fwd(qr[:1, :n], kr[:1, :n], idr[:1, :n], posr[:1, :n],
                                         window_left=window_left),
                     dtype=torch.uint8, device=dev)
    for bi in range(b):
        for r in range(R):
            rows = slice(r * n, (r + 1) * n)
            qv, iq, pq = qr[bi:bi + 1, rows], idr[bi:bi + 1, rows], posr[bi:bi + 1, rows]
            lacc = lse_sh[r:r + 1]
            for t in range(R):
                j = (r - t) % R
                cols = slice(j * n, (j + 1) * n)
                kv = (kr[bi:bi + 1, cols], vr[bi:bi + 1, cols], idr[bi:bi + 1, cols],
                      posr[bi:bi + 1, cols])
                if R == 1:
                    attn_fwd(qv, kv[0], kv[1], iq, pq, kv[2], kv[3], window_left=window_left,
                             scale=scale, out=out_r[:, rows], lse=lacc, workspace=ws)
                elif t == 0:
                    attn_fwd(qv, kv[0], kv[1], iq, pq, kv[2], kv[3], window_left=window_left,
                             scale=scale, out=acc, lse=lacc, out_fp32=True, workspace=ws)
                else:
                    attn_fwd(qv, kv[0], kv[1], iq, pq, kv[2], kv[3], window_left=window_left,
                             scale=scale, out=blk, lse=blk_lse, out_fp32=True, workspace=ws)
                    attn_merge_partial(acc, lacc, blk, blk_lse,
                                       out_final=out_r[:, rows] if t == R - 1 else None)
        # [R, Hq, n] -> [Hq, R*n]: a block transpose, done as a striped permutation
        # of R*Hq stripes of n values over Hq logical shards.
        lse_t = reorder_causal_lb(lse_sh.view(1, R * hq * n), STRIPED, hq, n, seq_dim=1)
        inverse_reorder_causal_lb(lse_t.view(hq, s), strategy, R, stripe_size, seq_dim=1,
                                  out=lse[bi])
        inverse_reorder_causal_lb(out_r, strategy, R, stripe_size, seq_dim=1,
                                  out=out[bi:bi + 1])
    return out, lse
