"""gb300attn: exact packed-THD attention for one GB300 (sm_103a).

Thin ctypes binding over the C ABI in ``include/gb300attn.h``.  This module
only marshals arguments (tensor pointers, sizes, the current CUDA stream) and
allocates result tensors with PyTorch; every step of the computation runs in
the library's CUDA kernels.  There is no CPU fallback: every call raises if
the shared library is missing or a tensor is not on a CUDA device.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgb300attn.so")

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = range(5)
DUAL_CHUNK, STRIPED = 0, 1
TILE = 128

EXPORTS = (
    "attn_fwd_workspace_bytes", "attn_bwd_workspace_bytes", "attn_fwd", "attn_bwd",
    "attn_merge_partial", "reorder_causal_lb", "inverse_reorder_causal_lb", "attn_tile_plan",
    "attn_read_device_status", "attn_status_string", "attn_fwd_noalloc",
    "attn_fwd_test_timeout", "attn_segments_from_seqlens", "attn_fwd_noalloc_status",
    "attn_tile_order",
)


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} (status {code})")
        self.code = code


class FwdParams(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("q_segment_ids", ctypes.c_void_p), ("q_segment_pos", ctypes.c_void_p),
        ("kv_segment_ids", ctypes.c_void_p), ("kv_segment_pos", ctypes.c_void_p),
        ("b", ctypes.c_int64), ("s_q", ctypes.c_int64), ("s_kv", ctypes.c_int64),
        ("h_q", ctypes.c_int64), ("h_kv", ctypes.c_int64), ("d", ctypes.c_int64),
        ("window_left", ctypes.c_int32), ("window_right", ctypes.c_int32),
        ("scale", ctypes.c_float), ("out_fp32", ctypes.c_int32),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("merge_into_out", ctypes.c_int32), ("out_final", ctypes.c_void_p),
        ("kv_token_stride", ctypes.c_int64), ("d_v", ctypes.c_int64),
    ]


class BwdParams(ctypes.Structure):
    _fields_ = [
        ("fwd", FwdParams), ("dout", ctypes.c_void_p), ("dq", ctypes.c_void_p),
        ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p), ("accumulate_fp32", ctypes.c_int32),
        ("deterministic", ctypes.c_int32), ("kernel_events", ctypes.c_void_p * 2),
        ("delta", ctypes.c_void_p),
    ]


_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it has not been built)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        h = ctypes.CDLL(LIB_PATH)
        vp, i64, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        h.attn_fwd_workspace_bytes.argtypes = [ctypes.POINTER(FwdParams)]
        h.attn_fwd_workspace_bytes.restype = ctypes.c_size_t
        h.attn_bwd_workspace_bytes.argtypes = [ctypes.POINTER(BwdParams)]
        h.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        h.attn_fwd.argtypes = [ctypes.POINTER(FwdParams), vp]
        h.attn_fwd.restype = c_int
        h.attn_bwd.argtypes = [ctypes.POINTER(BwdParams), vp]
        h.attn_bwd.restype = c_int
        h.attn_merge_partial.argtypes = [vp, vp, vp, vp, c_int, vp, i64, i64, i64, i64, vp]
        h.attn_merge_partial.restype = c_int
        for name in ("reorder_causal_lb", "inverse_reorder_causal_lb"):
            f = getattr(h, name)
            f.argtypes = [vp, vp, i64, i64, i64, c_int, c_int, c_int, vp]
            f.restype = c_int
        h.attn_tile_plan.argtypes = [ctypes.POINTER(FwdParams), vp, vp, vp]
        h.attn_tile_plan.restype = c_int
        h.attn_tile_order.argtypes = [ctypes.POINTER(FwdParams), vp, vp, vp]
        h.attn_tile_order.restype = c_int
        h.attn_read_device_status.argtypes = [vp, vp]
        h.attn_read_device_status.restype = c_int
        h.attn_fwd_test_timeout.argtypes = [ctypes.POINTER(FwdParams), vp]
        h.attn_fwd_test_timeout.restype = c_int
        h.attn_fwd_noalloc.argtypes = [ctypes.POINTER(FwdParams), vp]
        h.attn_fwd_noalloc.restype = c_int
        h.attn_fwd_noalloc_status.argtypes = [vp]
        h.attn_fwd_noalloc_status.restype = c_int
        h.attn_segments_from_seqlens.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp]
        h.attn_segments_from_seqlens.restype = c_int
        h.attn_status_string.argtypes = [c_int]
        h.attn_status_string.restype = ctypes.c_char_p
        _lib_handle = h
    return _lib_handle


def status_string(code: int) -> str:
    return lib().attn_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != ATTN_OK:
        raise AttnError(code, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("gb300attn runs on CUDA tensors only")
        if t is not None and not t.is_contiguous():
            raise ValueError("gb300attn expects contiguous tensors")


def _kv_token_stride(*ts) -> int:
    """Token stride (elements) shared by k / v-shaped tensors [b, s, h, d]
    that may be views into a packed K/V tensor [b, s, 2, h, d] (THD_T2HD);
    0 when they are contiguous."""
    ref = ts[0]
    b, s, h, d = ref.shape
    for t in ts:
        if not t.is_cuda:
            raise ValueError("gb300attn runs on CUDA tensors only")
        if t.shape != ref.shape or t.stride() != ref.stride():
            raise ValueError("k and v (and dk, dv) must share one shape and layout")
    st = ref.stride()
    if st[3] != 1 or (h > 1 and st[2] != d):
        raise ValueError("k / v: heads and head dims must be contiguous")
    ts_ = st[1] if s > 1 else h * d
    if ts_ < h * d or (b > 1 and st[0] != s * ts_):
        raise ValueError("k / v: unsupported token or batch stride")
    return 0 if ts_ == h * d else int(ts_)


def _fwd_params(q, k, v, q_ids, q_pos, kv_ids, kv_pos, window_left, scale, out, lse, out_fp32):
    b, s_q, hq, d = q.shape
    _, s_kv, hkv, _ = k.shape
    p = FwdParams()
    p.q, p.k, p.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    p.q_segment_ids, p.q_segment_pos = q_ids.data_ptr(), q_pos.data_ptr()
    p.kv_segment_ids, p.kv_segment_pos = kv_ids.data_ptr(), kv_pos.data_ptr()
    p.b, p.s_q, p.s_kv, p.h_q, p.h_kv, p.d = b, s_q, s_kv, hq, hkv, d
    p.d_v = v.shape[3] if v.shape[3] != d else 0  # 0: V has the head dim of q and k
    p.window_left, p.window_right = int(window_left), 0
    p.scale = float(d ** -0.5 if scale is None else scale)
    p.out_fp32 = 1 if out_fp32 else 0
    p.out = out.data_ptr() if out is not None else None
    p.lse = lse.data_ptr() if lse is not None else None
    return p


def workspace_bytes_fwd(q, k, q_ids, q_pos, kv_ids=None, kv_pos=None, window_left=-1,
                        scale=None, v=None) -> int:
    """Workspace bytes attn_fwd needs for these shapes (0 if it rejects them);
    pass ``v`` when its head dim differs from k's."""
    kv_ids = q_ids if kv_ids is None else kv_ids
    kv_pos = q_pos if kv_pos is None else kv_pos
    v = k if v is None else v
    p = _fwd_params(q, k, v, q_ids, q_pos, kv_ids, kv_pos, window_left, scale, q, q, False)
    return int(lib().attn_fwd_workspace_bytes(ctypes.byref(p)))


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def attn_fwd(q, k, v, q_ids, q_pos, kv_ids=None, kv_pos=None, *, window_left: int = -1,
             scale: Optional[float] = None, out=None, lse=None, out_fp32: bool = False,
             merge_into_out: bool = False, out_final=None,
             workspace: Optional[torch.Tensor] = None, check_status: bool = False):
    """Forward attention.  Returns (out [b,s_q,Hq,d_v], lse fp32 [b,Hq,s_q]).

    q bf16 [b,s_q,Hq,d]; k bf16 [b,s_kv,Hkv,d]; v bf16 [b,s_kv,Hkv,d_v] (d_v = d,
    or d = 192 with d_v = 128); ids/pos int32 [b,s].
    kv_ids / kv_pos default to the query descriptor (self-attention).
    With ``merge_into_out`` the given fp32 ``out`` / ``lse`` hold a finished
    partial over other key blocks and this call's result is merged into them
    (into bf16 ``out_final`` instead of ``out`` when given).
    ``check_status`` synchronises the stream after the launch and raises
    :class:`AttnError` (``ATTN_ERR_TIMEOUT``) if a bounded device-side wait gave
    up, in which case the outputs are undefined; otherwise the call stays
    asynchronous and the status can be read later from ``workspace`` with
    :func:`read_device_status`.
    """
    return _attn_fwd_call("attn_fwd", q, k, v, q_ids, q_pos, kv_ids, kv_pos, window_left, scale,
                          out, lse, out_fp32, merge_into_out, out_final, workspace, check_status)


def attn_fwd_test_timeout(q, k, v, q_ids, q_pos, kv_ids=None, kv_pos=None, *,
                          window_left: int = -1, scale: Optional[float] = None,
                          workspace: Optional[torch.Tensor] = None, check_status: bool = True):
    """Test hook: attn_fwd with every key / value load withheld, so the
    device-side waits run out (about a second) and the launch records
    ``ATTN_ERR_TIMEOUT``; with ``check_status`` (the default) that raises
    :class:`AttnError` here.  Not for production use."""
    return _attn_fwd_call("attn_fwd_test_timeout", q, k, v, q_ids, q_pos, kv_ids, kv_pos,
                          window_left, scale, None, None, False, False, None, workspace,
                          check_status)


def _raise_on_device_status(workspace: torch.Tensor, what: str):
    code = read_device_status(workspace)
    if code != ATTN_OK:
        raise AttnError(code, what)


def _attn_fwd_call(entry, q, k, v, q_ids, q_pos, kv_ids, kv_pos, window_left, scale, out, lse,
                   out_fp32, merge_into_out, out_final, workspace, check_status):
    kv_ids = q_ids if kv_ids is None else kv_ids
    kv_pos = q_pos if kv_pos is None else kv_pos
    _need_cuda(q, q_ids, q_pos, kv_ids, kv_pos, out, lse, workspace, out_final)
    if v.shape[3] != k.shape[3]:
        # V narrower or wider than Q / K (d_qk != d_v): separate, contiguous tensors
        if not (k.is_contiguous() and v.is_contiguous()) or v.shape[:3] != k.shape[:3]:
            raise ValueError("k / v of different head dims must be contiguous [b, s, h, d]")
        kv_stride = 0
    else:
        kv_stride = _kv_token_stride(k, v)
    if merge_into_out and (out is None or lse is None or not out_fp32):
        raise ValueError("merge_into_out needs the fp32 out and lse accumulators")
    b, s_q, hq, _ = q.shape
    d = v.shape[3]  # the output has V's head dim
    if out is None:
        out = torch.empty(b, s_q, hq, d, device=q.device,
                          dtype=torch.float32 if out_fp32 else torch.bfloat16)
    if lse is None:
        lse = torch.empty(b, hq, s_q, device=q.device, dtype=torch.float32)
    p = _fwd_params(q, k, v, q_ids, q_pos, kv_ids, kv_pos, window_left, scale, out, lse, out_fp32)
    p.merge_into_out = 1 if merge_into_out else 0
    p.out_final = out_final.data_ptr() if out_final is not None else None
    p.kv_token_stride = kv_stride
    need = lib().attn_fwd_workspace_bytes(ctypes.byref(p))
    if workspace is None:
        workspace = _workspace(need, q.device)
    p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    _check(getattr(lib(), entry)(ctypes.byref(p), _stream(q.device)), entry)
    if check_status:
        _raise_on_device_status(workspace, entry)
    return out, lse


def attn_bwd(q, k, v, out, lse, dout, q_ids, q_pos, kv_ids=None, kv_pos=None, *,
             window_left: int = -1, scale: Optional[float] = None, dq=None, dk=None, dv=None,
             accumulate_fp32: bool = False, workspace: Optional[torch.Tensor] = None,
             check_status: bool = False, deterministic: bool = False, kernel_events=None,
             delta=None):
    """Backward attention.  Returns (dq, dk, dv): bf16, or with
    ``accumulate_fp32`` the given fp32 tensors with this call's gradients added.
    ``deterministic`` takes the dK / dV + dQ kernel pair, whose results are
    bit-identical from run to run (the default fused kernel sums dQ with
    reduce-adds in hardware order); head dims 256 and (192, 128) always take it.
    ``kernel_events`` (two timing ``torch.cuda.Event``) are recorded just
    before and after the main kernel(s), without the plan, the D pre-pass and
    the dQ finalise.  ``delta`` (fp32 [b, Hq, s_q], optional) receives
    D = rowsum(dO * O) of every query row and head; its sum is vdot(out,
    dout), the loss whose gradient this call computes.  ``check_status`` as in
    :func:`attn_fwd`."""
    kv_ids = q_ids if kv_ids is None else kv_ids
    kv_pos = q_pos if kv_pos is None else kv_pos
    _need_cuda(q, out, lse, dout, q_ids, q_pos, kv_ids, kv_pos, workspace, dq)
    mla = v.shape[3] != k.shape[3]
    if mla:
        # V narrower than Q / K (d_qk 192, d_v 128): separate, contiguous tensors
        _need_cuda(k, v, dk, dv)
        if v.shape[:3] != k.shape[:3]:
            raise ValueError("k / v of different head dims must share [b, s, h]")
        kv_stride = 0
    else:
        kv_stride = _kv_token_stride(k, v)
    if kv_stride and (dk is None or dv is None):
        if kv_stride != 2 * k.shape[2] * k.shape[3]:
            raise ValueError("strided k / v: pass dk and dv in the same layout")
        dkv = torch.empty(k.shape[0], k.shape[1], 2, k.shape[2], k.shape[3], device=k.device,
                          dtype=torch.float32 if accumulate_fp32 else k.dtype)
        dk, dv = (dkv[:, :, 0] if dk is None else dk), (dkv[:, :, 1] if dv is None else dv)
    if accumulate_fp32:
        if dq is None or dk is None or dv is None:
            raise ValueError("accumulate_fp32 needs fp32 dq, dk and dv accumulators")
        if not all(t.dtype == torch.float32 for t in (dq, dk, dv)):
            raise ValueError("accumulate_fp32 needs fp32 dq, dk and dv accumulators")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if mla:
        if dk.shape != k.shape or dv.shape != v.shape:
            raise ValueError("dk / dv must have the shapes of k / v")
    else:
        _kv_token_stride(k, v, dk, dv)  # dk / dv must have the layout of k / v
    p = BwdParams()
    p.fwd = _fwd_params(q, k, v, q_ids, q_pos, kv_ids, kv_pos, window_left, scale, out, lse, False)
    p.fwd.kv_token_stride = kv_stride
    p.dout, p.dq, p.dk, p.dv = dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    p.accumulate_fp32 = 1 if accumulate_fp32 else 0
    p.deterministic = 1 if deterministic else 0
    if delta is not None:
        _need_cuda(delta)
        if delta.dtype != torch.float32 or delta.shape != (q.shape[0], q.shape[2], q.shape[1]):
            raise ValueError("delta must be a contiguous fp32 [b, Hq, s_q] tensor")
        p.delta = delta.data_ptr()
    if kernel_events is not None:
        for i, ev in enumerate(kernel_events):
            if not ev.cuda_event:  # a torch event exists once it has been recorded
                ev.record(torch.cuda.current_stream(q.device))
            p.kernel_events[i] = ev.cuda_event
    need = lib().attn_bwd_workspace_bytes(ctypes.byref(p))
    if workspace is None:
        workspace = _workspace(need, q.device)
    p.fwd.workspace, p.fwd.workspace_bytes = workspace.data_ptr(), workspace.numel()
    _check(lib().attn_bwd(ctypes.byref(p), _stream(q.device)), "attn_bwd")
    if check_status:
        _raise_on_device_status(workspace, "attn_bwd")
    return dq, dk, dv


def workspace_bytes_bwd(q, k, q_ids, q_pos, window_left=-1, v=None,
                        deterministic: bool = False) -> int:
    """Workspace bytes attn_bwd needs for these shapes (0 if it rejects them);
    pass ``v`` when its head dim differs from k's."""
    p = BwdParams()
    p.fwd = _fwd_params(q, k, k if v is None else v, q_ids, q_pos, q_ids, q_pos, window_left,
                        None, q, q, False)
    p.deterministic = 1 if deterministic else 0
    return int(lib().attn_bwd_workspace_bytes(ctypes.byref(p)))


def segments_from_seqlens(seqlens, s: int, offsets=None):
    """Segment ids / pos int32 [b, s] from lengths int32 [b, nseg] (and start
    offsets [b, nseg]; None = segments back to back), on the lengths' device."""
    _need_cuda(seqlens, offsets)
    if seqlens.dim() != 2 or seqlens.dtype != torch.int32 or not seqlens.is_contiguous():
        raise ValueError("seqlens must be a contiguous int32 [b, nseg] tensor")
    if offsets is not None and (offsets.shape != seqlens.shape or offsets.dtype != torch.int32
                                or not offsets.is_contiguous()):
        raise ValueError("offsets must be a contiguous int32 tensor shaped like seqlens")
    b, nseg = seqlens.shape
    ids = torch.empty(b, s, dtype=torch.int32, device=seqlens.device)
    pos = torch.empty(b, s, dtype=torch.int32, device=seqlens.device)
    _check(lib().attn_segments_from_seqlens(
        seqlens.data_ptr(), offsets.data_ptr() if offsets is not None else None, b, nseg, s,
        ids.data_ptr(), pos.data_ptr(), _stream(seqlens.device)), "attn_segments_from_seqlens")
    return ids, pos


def attn_merge_partial(out_acc, lse_acc, out_blk, lse_blk, out_final=None):
    """Online-softmax merge of (out_blk, lse_blk) into (out_acc, lse_acc), in place.

    out_acc fp32 [b,s,H,d]; lse_* fp32 [b,H,s]; out_blk fp32 or bf16.
    With ``out_final`` (bf16 [b,s,H,d]) the merged output goes there instead.
    """
    _need_cuda(out_acc, lse_acc, out_blk, lse_blk, out_final)
    b, s, h, d = out_acc.shape
    rc = lib().attn_merge_partial(
        _ptr(out_acc), _ptr(lse_acc), _ptr(out_blk), _ptr(lse_blk),
        1 if out_blk.dtype == torch.bfloat16 else 0, _ptr(out_final), b, s, h, d,
        _stream(out_acc.device))
    _check(rc, "attn_merge_partial")
    return (out_final if out_final is not None else out_acc), lse_acc


def _seq_view(x: torch.Tensor, seq_dim: int):
    outer = 1
    for n in x.shape[:seq_dim]:
        outer *= n
    inner = x.element_size()
    for n in x.shape[seq_dim + 1:]:
        inner *= n
    return outer, x.shape[seq_dim], inner


def reorder_causal_lb(x, strategy: int = DUAL_CHUNK, cp_size: int = 4, stripe_size: int = 1,
                      seq_dim: int = 1, out=None):
    """Causal load-balancing reorder along ``seq_dim`` (returns a new tensor)."""
    _need_cuda(x, out)
    out = torch.empty_like(x) if out is None else out
    outer, s, inner = _seq_view(x, seq_dim)
    rc = lib().reorder_causal_lb(_ptr(x), _ptr(out), outer, s, inner, strategy, cp_size,
                                 stripe_size, _stream(x.device))
    _check(rc, "reorder_causal_lb")
    return out


def inverse_reorder_causal_lb(x, strategy: int = DUAL_CHUNK, cp_size: int = 4,
                              stripe_size: int = 1, seq_dim: int = 1, out=None):
    """Inverse of :func:`reorder_causal_lb` with the same arguments."""
    _need_cuda(x, out)
    out = torch.empty_like(x) if out is None else out
    outer, s, inner = _seq_view(x, seq_dim)
    rc = lib().inverse_reorder_causal_lb(_ptr(x), _ptr(out), outer, s, inner, strategy, cp_size,
                                         stripe_size, _stream(x.device))
    _check(rc, "inverse_reorder_causal_lb")
    return out


def attn_tile_plan(q, k, q_ids, q_pos, kv_ids=None, kv_pos=None, *, window_left: int = -1,
                   workspace=None):
    """Per-tile classes (uint8 [b,nq,nk]: 0 SKIP, 1 PARTIAL, 2 FULL) and q ranges."""
    kv_ids = q_ids if kv_ids is None else kv_ids
    kv_pos = q_pos if kv_pos is None else kv_pos
    _need_cuda(q, k, q_ids, q_pos, kv_ids, kv_pos)
    b, s_q = q.shape[:2]
    s_kv = k.shape[1]
    nq, nk = -(-s_q // TILE), -(-s_kv // TILE)
    p = _fwd_params(q, k, k, q_ids, q_pos, kv_ids, kv_pos, window_left, None, q, q, False)
    need = lib().attn_fwd_workspace_bytes(ctypes.byref(p))
    workspace = _workspace(need, q.device) if workspace is None else workspace
    p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    cls = torch.empty(b, nq, nk, dtype=torch.uint8, device=q.device)
    rng = torch.empty(b, nq, 2, dtype=torch.int32, device=q.device)
    _check(lib().attn_tile_plan(ctypes.byref(p), _ptr(cls), _ptr(rng), _stream(q.device)),
           "attn_tile_plan")
    return cls, rng


def attn_tile_order(q, k, q_ids, q_pos, kv_ids=None, kv_pos=None, *, window_left: int = -1,
                    workspace=None):
    """The kernels' work order (debug hook): (q_order int32 [b*nq], kv_order
    int32 [b*nk]) as the forward and the fused backward take their units:
    index order (descending on the query side) when the heaviest unit is a
    small share of the launch, else a stable heaviest-first permutation."""
    kv_ids = q_ids if kv_ids is None else kv_ids
    kv_pos = q_pos if kv_pos is None else kv_pos
    _need_cuda(q, k, q_ids, q_pos, kv_ids, kv_pos)
    b, s_q = q.shape[:2]
    s_kv = k.shape[1]
    nq, nk = -(-s_q // TILE), -(-s_kv // TILE)
    p = _fwd_params(q, k, k, q_ids, q_pos, kv_ids, kv_pos, window_left, None, q, q, False)
    need = lib().attn_fwd_workspace_bytes(ctypes.byref(p))
    workspace = _workspace(need, q.device) if workspace is None else workspace
    p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    qo = torch.empty(b * nq, dtype=torch.int32, device=q.device)
    ko = torch.empty(b * nk, dtype=torch.int32, device=q.device)
    _check(lib().attn_tile_order(ctypes.byref(p), _ptr(qo), _ptr(ko), _stream(q.device)),
           "attn_tile_order")
    return qo, ko


def read_device_status(workspace: torch.Tensor) -> int:
    """Synchronise the current stream and read the device status word."""
    return int(lib().attn_read_device_status(_ptr(workspace), _stream(workspace.device)))


def noalloc_status() -> int:
    """Synchronise the current stream and read the status word of
    attn_fwd_noalloc's built-in scratch on the current device."""
    dev = torch.cuda.current_device()
    return int(lib().attn_fwd_noalloc_status(_stream(dev)))
