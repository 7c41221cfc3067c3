"""Context parallelism (ring and all-gather) emulated on one GPU.

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
attn_fwd on shard views (fp32 partial output) with the merge folded into its
epilogue, or attn_merge_partial as a separate pass.  This module is host
control only.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (ATTN_OK, DUAL_CHUNK, STRIPED, AttnError, attn_bwd, attn_fwd, attn_merge_partial,
               inverse_reorder_causal_lb, reorder_causal_lb, workspace_bytes_bwd,
               workspace_bytes_fwd)


class _StatusLog:
    """The device status word of every attention call of a driver run.

    Each call clears its workspace's status word when it starts, so the word
    is copied aside (a 4-byte device-to-device copy, no kernel) after every
    call and all copies are read once, with one synchronisation, at the end."""

    def __init__(self, n: int, device):
        self.words = torch.zeros(max(n, 1), dtype=torch.int32, device=device)
        self.n = 0

    def record(self, ws: torch.Tensor):
        self.words[self.n:self.n + 1].copy_(ws[:4].view(torch.int32))
        self.n += 1

    def check(self, what: str):
        worst = int(self.words[:self.n].max().item()) if self.n else ATTN_OK
        if worst != ATTN_OK:
            raise AttnError(worst, what)


def ring_attn_fwd(q, k, v, ids, pos, cp_size: int, *, window_left: int = -1,
                  scale: Optional[float] = None, strategy: int = DUAL_CHUNK, stripe_size: int = 1,
                  fused_merge: bool = True, check_status: bool = True,
                  batch_shards: bool = False):
    """Forward attention computed as cp_size ring steps per logical shard.

    q bf16 [b,s,Hq,d]; k, v bf16 [b,s,Hkv,d]; ids/pos int32 [b,s] (natural
    order).  Returns (out bf16 [b,s,Hq,d], lse fp32 [b,Hq,s]) in natural order.
    ``fused_merge`` folds each step's partial into the running result in the
    attention kernel's epilogue; otherwise a separate merge pass runs per step.
    ``check_status`` reads every call's device status word once at the end
    (one synchronisation) and raises :class:`AttnError` if a bounded
    device-side wait gave up, rather than returning undefined output.
    ``batch_shards`` runs each ring step as one call over all shards (the
    shards' queries as a batch of b*R rows, the K/V blocks they hold at that
    step rotated into place, as a ring's send / receive would move them)
    instead of one call per shard and step; the result is the same.
    """
    b, s, hq, d = q.shape
    dv = v.shape[3]  # the output takes V's head dim
    R = int(cp_size)
    if s % R:
        raise ValueError("sequence length must be divisible by cp_size")
    n = s // R
    dev = q.device
    re = lambda x: reorder_causal_lb(x, strategy, R, stripe_size, seq_dim=1)
    qr, kr, vr, idr, posr = re(q), re(k), re(v), re(ids), re(pos)
    if batch_shards:
        return _ring_fwd_batched(qr, kr, vr, idr, posr, R, window_left, scale, strategy,
                                 stripe_size, fused_merge, check_status, dv)
    out = torch.empty(b, s, hq, dv, dtype=q.dtype, device=dev)
    lse = torch.empty(b, hq, s, dtype=torch.float32, device=dev)
    acc = torch.empty(1, n, hq, dv, dtype=torch.float32, device=dev)
    blk = torch.empty(1, n, hq, dv, dtype=torch.float32, device=dev)
    blk_lse = torch.empty(1, hq, n, dtype=torch.float32, device=dev)
    lse_sh = torch.empty(R, hq, n, dtype=torch.float32, device=dev)
    out_r = torch.empty(1, s, hq, dv, dtype=q.dtype, device=dev)
    ws = torch.empty(workspace_bytes_fwd(qr[:1, :n], kr[:1, :n], idr[:1, :n], posr[:1, :n],
                                         window_left=window_left, v=vr[:1, :n]),
                     dtype=torch.uint8, device=dev)
    log = _StatusLog(b * R * R, dev) if check_status else None
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
                elif fused_merge:
                    attn_fwd(qv, kv[0], kv[1], iq, pq, kv[2], kv[3], window_left=window_left,
                             scale=scale, out=acc, lse=lacc, out_fp32=True, merge_into_out=True,
                             out_final=out_r[:, rows] if t == R - 1 else None, workspace=ws)
                else:
                    attn_fwd(qv, kv[0], kv[1], iq, pq, kv[2], kv[3], window_left=window_left,
                             scale=scale, out=blk, lse=blk_lse, out_fp32=True, workspace=ws)
                    attn_merge_partial(acc, lacc, blk, blk_lse,
                                       out_final=out_r[:, rows] if t == R - 1 else None)
                if log is not None:
                    log.record(ws)
        # [R, Hq, n] -> [Hq, R*n]: a block transpose, done as a striped permutation
        # of R*Hq stripes of n values over Hq logical shards.
        lse_t = reorder_causal_lb(lse_sh.view(1, R * hq * n), STRIPED, hq, n, seq_dim=1)
        inverse_reorder_causal_lb(lse_t.view(hq, s), strategy, R, stripe_size, seq_dim=1,
                                  out=lse[bi])
        inverse_reorder_causal_lb(out_r, strategy, R, stripe_size, seq_dim=1,
                                  out=out[bi:bi + 1])
    if log is not None:
        log.check("ring_attn_fwd")
    return out, lse


def allgather_attn_fwd(q, k, v, ids, pos, cp_size: int, *, window_left: int = -1,
                       scale: Optional[float] = None, strategy: int = STRIPED,
                       stripe_size: int = 512, check_status: bool = True):
    """All-gather context parallelism on one GPU (TE tutorial section 5,
    "AllGather" with a striped reorder, stripe_size 512; "Context parallelism
    and ring attention", section "Communication choices").

    Each logical shard r keeps its query rows [r*s/R, (r+1)*s/R) of the
    reordered sequence and attends, in one attn_fwd call, to the whole
    reordered K/V (what an all-gather of K/V would give every device).  The
    mask uses the reordered segment positions, so the result equals full
    attention.  Returns (out bf16 [b,s,Hq,d], lse fp32 [b,Hq,s]) in natural
    token order.  ``check_status`` as in :func:`ring_attn_fwd`.
    """
    b, s, hq, d = q.shape
    dv = v.shape[3]
    R = int(cp_size)
    if s % R:
        raise ValueError("sequence length must be divisible by cp_size")
    n = s // R
    dev = q.device
    re = lambda x: reorder_causal_lb(x, strategy, R, stripe_size, seq_dim=1)
    qr, kr, vr, idr, posr = re(q), re(k), re(v), re(ids), re(pos)
    out = torch.empty(b, s, hq, dv, dtype=q.dtype, device=dev)
    lse = torch.empty(b, hq, s, dtype=torch.float32, device=dev)
    out_r = torch.empty(1, s, hq, dv, dtype=q.dtype, device=dev)
    lse_sh = torch.empty(R, hq, n, dtype=torch.float32, device=dev)
    ws = torch.empty(workspace_bytes_fwd(qr[:1, :n], kr[:1], idr[:1, :n], posr[:1, :n],
                                         idr[:1], posr[:1], window_left=window_left, v=vr[:1]),
                     dtype=torch.uint8, device=dev)
    log = _StatusLog(b * R, dev) if check_status else None
    for bi in range(b):
        kv = (kr[bi:bi + 1], vr[bi:bi + 1], idr[bi:bi + 1], posr[bi:bi + 1])
        for r in range(R):
            rows = slice(r * n, (r + 1) * n)
            attn_fwd(qr[bi:bi + 1, rows], kv[0], kv[1], idr[bi:bi + 1, rows],
                     posr[bi:bi + 1, rows], kv[2], kv[3], window_left=window_left, scale=scale,
                     out=out_r[:, rows], lse=lse_sh[r:r + 1], workspace=ws)
            if log is not None:
                log.record(ws)
        lse_t = reorder_causal_lb(lse_sh.view(1, R * hq * n), STRIPED, hq, n, seq_dim=1)
        inverse_reorder_causal_lb(lse_t.view(hq, s), strategy, R, stripe_size, seq_dim=1,
                                  out=lse[bi])
        inverse_reorder_causal_lb(out_r, strategy, R, stripe_size, seq_dim=1,
                                  out=out[bi:bi + 1])
    if log is not None:
        log.check("allgather_attn_fwd")
    return out, lse


def ring_attn_bwd(q, k, v, out, lse, dout, ids, pos, cp_size: int, *, window_left: int = -1,
                  scale: Optional[float] = None, strategy: int = DUAL_CHUNK,
                  stripe_size: int = 1, check_status: bool = True,
                  deterministic: bool = False, batch_shards: bool = False):
    """Backward of ring attention, emulated on one GPU.

    Shard r keeps its query rows, final output O_r, LSE_r and dO_r; at step t
    it meets key/value block j = (r - t) mod R and adds that block's share of
    the gradient: dQ_r += dS_rj K_j, dK_j += dS_rj^T Q_r, dV_j += P_rj^T dO_r,
    with P_rj = exp(scale Q_r K_j^T - LSE_r) from the FINAL LSE and
    dS_rj = P_rj * (dP_rj - D_r), D_r = rowsum(dO_r * O_r) from the final output
    ("Context parallelism and ring attention", sections "Ring attention" and
    "Online softmax": the blocks' softmax pieces share one denominator).  Every
    contribution is accumulated in fp32 by attn_bwd's accumulate mode.

    out / lse: the forward results in natural order (e.g. from ring_attn_fwd).
    Returns fp32 (dq [b,s,Hq,d], dk, dv [b,s,Hkv,d]) in natural order.
    ``check_status`` as in :func:`ring_attn_fwd`; ``deterministic`` as in
    :func:`attn_bwd` (the block calls then add fixed-order sums, so the
    result is bit-identical from run to run).  ``batch_shards`` runs each ring
    step as one call over all shards, with the K/V blocks and their dK / dV
    accumulators rotated one shard on between steps (a ring moves the dK / dV
    partial sums along with the blocks); dK / dV are then summed over the
    shards in another order, equal within fp32 rounding.
    """
    b, s, hq, d = q.shape
    hkv = k.shape[2]
    R = int(cp_size)
    if s % R:
        raise ValueError("sequence length must be divisible by cp_size")
    n = s // R
    dev = q.device
    re = lambda x: reorder_causal_lb(x, strategy, R, stripe_size, seq_dim=1)
    qr, kr, vr, outr, dor = re(q), re(k), re(v), re(out), re(dout)
    idr, posr = re(ids), re(pos)
    if batch_shards:
        return _ring_bwd_batched(qr, kr, vr, outr, dor, idr, posr, lse, R, window_left, scale,
                                 strategy, stripe_size, check_status, deterministic)
    dq = torch.zeros(b, s, hq, d, dtype=torch.float32, device=dev)
    dk = torch.zeros(b, s, hkv, d, dtype=torch.float32, device=dev)
    dv = torch.zeros(b, s, hkv, v.shape[3], dtype=torch.float32, device=dev)
    lse_sh = torch.empty(R, hq, n, dtype=torch.float32, device=dev)
    ws = torch.empty(workspace_bytes_bwd(qr[:1, :n], kr[:1, :n], idr[:1, :n], posr[:1, :n],
                                         window_left, v=vr[:1, :n],
                                         deterministic=deterministic),
                     dtype=torch.uint8, device=dev)
    log = _StatusLog(b * R * R, dev) if check_status else None
    for bi in range(b):
        # this row's LSE in reordered order, then [Hq, R*n] -> [R, Hq, n] so that
        # every shard's LSE is contiguous (the inverse of a striped block transpose)
        lse_r = reorder_causal_lb(lse[bi], strategy, R, stripe_size, seq_dim=1)
        inverse_reorder_causal_lb(lse_r.view(1, hq * s), STRIPED, hq, n, seq_dim=1,
                                  out=lse_sh.view(1, R * hq * n))
        for r in range(R):
            rq = slice(r * n, (r + 1) * n)
            for t in range(R):
                j = (r - t) % R
                rk = slice(j * n, (j + 1) * n)
                attn_bwd(qr[bi:bi + 1, rq], kr[bi:bi + 1, rk], vr[bi:bi + 1, rk],
                         outr[bi:bi + 1, rq], lse_sh[r:r + 1], dor[bi:bi + 1, rq],
                         idr[bi:bi + 1, rq], posr[bi:bi + 1, rq], idr[bi:bi + 1, rk],
                         posr[bi:bi + 1, rk], window_left=window_left, scale=scale,
                         dq=dq[bi:bi + 1, rq], dk=dk[bi:bi + 1, rk], dv=dv[bi:bi + 1, rk],
                         accumulate_fp32=True, workspace=ws, deterministic=deterministic)
                if log is not None:
                    log.record(ws)
    if log is not None:
        log.check("ring_attn_bwd")
    inv = lambda x: inverse_reorder_causal_lb(x, strategy, R, stripe_size, seq_dim=1)
    return inv(dq), inv(dk), inv(dv)


def allgather_attn_bwd(q, k, v, out, lse, dout, ids, pos, cp_size: int, *,
                       window_left: int = -1, scale: Optional[float] = None,
                       strategy: int = STRIPED, stripe_size: int = 512,
                       check_status: bool = True, deterministic: bool = False):
    """Backward of all-gather context parallelism, emulated on one GPU (TE
    tutorial section 5, "AllGather"; "Context parallelism and ring attention",
    section "Communication choices").

    Shard r keeps its query rows, final output O_r, LSE_r and dO_r of the
    reordered sequence and meets the whole reordered K/V (its all-gathered
    copy) in one attn_bwd call: that call gives dQ_r in full and adds the
    shard's share of dK and dV into accumulators over the whole sequence (on a
    mesh, a reduce-scatter of those accumulators returns every device its own
    rows).  P uses the final LSE and D = rowsum(dO * O) the final output, so
    the sum over shards is the full gradient.  Returns (dq, dk, dv) fp32 in
    natural token order.  ``check_status`` and ``deterministic`` as in
    :func:`ring_attn_bwd`.
    """
    b, s, hq, d = q.shape
    R = int(cp_size)
    if s % R:
        raise ValueError("sequence length must be divisible by cp_size")
    n = s // R
    dev = q.device
    re = lambda x: reorder_causal_lb(x, strategy, R, stripe_size, seq_dim=1)
    qr, kr, vr, outr, dor = re(q), re(k), re(v), re(out), re(dout)
    idr, posr = re(ids), re(pos)
    dq = torch.zeros(b, s, hq, d, dtype=torch.float32, device=dev)
    dk = torch.zeros(b, s, k.shape[2], d, dtype=torch.float32, device=dev)
    dv = torch.zeros(b, s, k.shape[2], v.shape[3], dtype=torch.float32, device=dev)
    lse_sh = torch.empty(R, hq, n, dtype=torch.float32, device=dev)
    ws = torch.empty(workspace_bytes_bwd(qr[:1, :n], kr[:1], idr[:1, :n], posr[:1, :n],
                                         window_left, v=vr[:1], deterministic=deterministic),
                     dtype=torch.uint8, device=dev)
    log = _StatusLog(b * R, dev) if check_status else None
    for bi in range(b):
        # this row's LSE in reordered order, then [Hq, R*n] -> [R, Hq, n]
        lse_r = reorder_causal_lb(lse[bi], strategy, R, stripe_size, seq_dim=1)
        inverse_reorder_causal_lb(lse_r.view(1, hq * s), STRIPED, hq, n, seq_dim=1,
                                  out=lse_sh.view(1, R * hq * n))
        kv = slice(bi, bi + 1)
        for r in range(R):
            rows = slice(r * n, (r + 1) * n)
            attn_bwd(qr[kv, rows], kr[kv], vr[kv], outr[kv, rows], lse_sh[r:r + 1], dor[kv, rows],
                     idr[kv, rows], posr[kv, rows], idr[kv], posr[kv], window_left=window_left,
                     scale=scale, dq=dq[kv, rows], dk=dk[kv], dv=dv[kv], accumulate_fp32=True,
                     workspace=ws, deterministic=deterministic)
            if log is not None:
                log.record(ws)
    if log is not None:
        log.check("allgather_attn_bwd")
    inv = lambda x: inverse_reorder_causal_lb(x, strategy, R, stripe_size, seq_dim=1)
    return inv(dq), inv(dk), inv(dv)



def _shard_lse(lse_rows, strategy, R, stripe_size, n):
    """[Hq, s] LSE of one batch row in natural order -> [R, Hq, n] by shard."""
    hq, s = lse_rows.shape
    lse_r = reorder_causal_lb(lse_rows, strategy, R, stripe_size, seq_dim=1)
    out = torch.empty(R, hq, n, dtype=torch.float32, device=lse_rows.device)
    inverse_reorder_causal_lb(lse_r.view(1, hq * s), STRIPED, hq, n, seq_dim=1,
                              out=out.view(1, R * hq * n))
    return out


def _natural_lse(lse_sh, strategy, R, stripe_size, out_row):
    """[R, Hq, n] LSE of one batch row by shard -> its [Hq, s] in natural order."""
    _, hq, n = lse_sh.shape
    lse_t = reorder_causal_lb(lse_sh.reshape(1, R * hq * n), STRIPED, hq, n, seq_dim=1)
    inverse_reorder_causal_lb(lse_t.view(hq, R * n), strategy, R, stripe_size, seq_dim=1,
                              out=out_row)


def _held_blocks(x, R, t):
    """The block every shard holds at ring step t, as a batch of b*R shards:
    shard r holds block (r - t) mod R of its batch row."""
    b, s = x.shape[:2]
    xs = x.reshape(b, R, s // R, *x.shape[2:])
    if t:
        xs = torch.roll(xs, shifts=t, dims=1)
    return xs.reshape(b * R, s // R, *x.shape[2:])


def _ring_fwd_batched(qr, kr, vr, idr, posr, R, window_left, scale, strategy, stripe_size,
                      fused_merge, check_status, dv):
    b, s, hq, d = qr.shape
    n = s // R
    B = b * R
    dev = qr.device
    qa, ida, pa = qr.view(B, n, hq, d), idr.view(B, n), posr.view(B, n)
    out_r = torch.empty(b, s, hq, dv, dtype=qr.dtype, device=dev)
    out_ra = out_r.view(B, n, hq, dv)
    lse_a = torch.empty(B, hq, n, dtype=torch.float32, device=dev)
    acc = torch.empty(B, n, hq, dv, dtype=torch.float32, device=dev)
    blk = torch.empty_like(acc) if not fused_merge else None
    blk_lse = torch.empty_like(lse_a) if not fused_merge else None
    ws = torch.empty(workspace_bytes_fwd(qa, kr.view(B, n, *kr.shape[2:]), ida, pa,
                                         window_left=window_left, v=vr.view(B, n, *vr.shape[2:])),
                     dtype=torch.uint8, device=dev)
    log = _StatusLog(R, dev) if check_status else None
    for t in range(R):
        kt, vt = _held_blocks(kr, R, t), _held_blocks(vr, R, t)
        it, pt = _held_blocks(idr, R, t), _held_blocks(posr, R, t)
        kw = dict(window_left=window_left, scale=scale, workspace=ws)
        if R == 1:
            attn_fwd(qa, kt, vt, ida, pa, it, pt, out=out_ra, lse=lse_a, **kw)
        elif t == 0:
            attn_fwd(qa, kt, vt, ida, pa, it, pt, out=acc, lse=lse_a, out_fp32=True, **kw)
        elif fused_merge:
            attn_fwd(qa, kt, vt, ida, pa, it, pt, out=acc, lse=lse_a, out_fp32=True,
                     merge_into_out=True, out_final=out_ra if t == R - 1 else None, **kw)
        else:
            attn_fwd(qa, kt, vt, ida, pa, it, pt, out=blk, lse=blk_lse, out_fp32=True, **kw)
            attn_merge_partial(acc, lse_a, blk, blk_lse, out_final=out_ra if t == R - 1 else None)
        if log is not None:
            log.record(ws)
    lse = torch.empty(b, hq, s, dtype=torch.float32, device=dev)
    for bi in range(b):
        _natural_lse(lse_a[bi * R:(bi + 1) * R], strategy, R, stripe_size, lse[bi])
    out = inverse_reorder_causal_lb(out_r, strategy, R, stripe_size, seq_dim=1)
    if log is not None:
        log.check("ring_attn_fwd")
    return out, lse


def _ring_bwd_batched(qr, kr, vr, outr, dor, idr, posr, lse, R, window_left, scale, strategy,
                      stripe_size, check_status, deterministic):
    b, s, hq, d = qr.shape
    hkv, dv = kr.shape[2], vr.shape[3]
    n = s // R
    B = b * R
    dev = qr.device
    qa, outa, doa = qr.view(B, n, hq, d), outr.view(B, n, hq, dv), dor.view(B, n, hq, dv)
    ida, pa = idr.view(B, n), posr.view(B, n)
    lse_a = torch.empty(B, hq, n, dtype=torch.float32, device=dev)
    for bi in range(b):
        lse_a[bi * R:(bi + 1) * R] = _shard_lse(lse[bi], strategy, R, stripe_size, n)
    dq = torch.zeros(b, s, hq, d, dtype=torch.float32, device=dev)
    # the dK / dV partial sums travel with their blocks: position r holds the
    # sums of block (r - t) mod R during step t
    dk_held = torch.zeros(b, s, hkv, d, dtype=torch.float32, device=dev)
    dv_held = torch.zeros(b, s, hkv, dv, dtype=torch.float32, device=dev)
    ws = torch.empty(workspace_bytes_bwd(qa, kr.view(B, n, hkv, d), ida, pa, window_left,
                                         v=vr.view(B, n, hkv, dv), deterministic=deterministic),
                     dtype=torch.uint8, device=dev)
    log = _StatusLog(R, dev) if check_status else None
    for t in range(R):
        kt, vt = _held_blocks(kr, R, t), _held_blocks(vr, R, t)
        it, pt = _held_blocks(idr, R, t), _held_blocks(posr, R, t)
        attn_bwd(qa, kt, vt, outa, lse_a, doa, ida, pa, it, pt, window_left=window_left,
                 scale=scale, dq=dq.view(B, n, hq, d), dk=dk_held.view(B, n, hkv, d),
                 dv=dv_held.view(B, n, hkv, dv), accumulate_fp32=True, workspace=ws,
                 deterministic=deterministic)
        if log is not None:
            log.record(ws)
        # pass the partial sums on with their blocks (after the last step every
        # block's sums are back at its own position)
        dk_held = _held_blocks(dk_held, R, 1).view(b, s, hkv, d)
        dv_held = _held_blocks(dv_held, R, 1).view(b, s, hkv, dv)
    if log is not None:
        log.check("ring_attn_bwd")
    inv = lambda x: inverse_reorder_causal_lb(x, strategy, R, stripe_size, seq_dim=1)
    return inv(dq), inv(dk_held), inv(dv_held)
