"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects invalid arguments on the host before touching
the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ga():
    import __graft_entry__
    __graft_entry__.build()
    import long_context_attention_attn_gb300 as pkg
    return pkg


def _header_symbols():
    with open(os.path.join(ROOT, "include", "gb300attn.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^GB300ATTN_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)))


def test_library_exports_every_declared_symbol(ga):
    syms = _header_symbols()
    assert len(syms) >= 10
    lib = ga.lib()
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) == set(ga.EXPORTS)


def test_status_strings(ga):
    assert ga.status_string(0) == "ok"
    assert "timed out" in ga.status_string(4)


def _params(ga, **kw):
    p = ga.FwdParams()
    fake = 1 << 20  # aligned non-null fake device address; never dereferenced
    for f in ("q", "k", "v", "q_segment_ids", "q_segment_pos", "kv_segment_ids",
              "kv_segment_pos", "out", "lse"):
        setattr(p, f, fake)
    p.workspace = fake
    p.b, p.s_q, p.s_kv, p.h_q, p.h_kv, p.d = 2, 4096, 4096, 16, 2, 128
    p.window_left, p.window_right, p.scale = -1, 0, 128 ** -0.5
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2), (dict(d=192), 2), (dict(window_right=1), 1), (dict(window_left=-2), 1),
    (dict(h_kv=3), 1), (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(b=0), 1),
    (dict(s_q=0), 1), (dict(q=None), 1), (dict(q=(1 << 20) + 8), 1), (dict(lse=None), 1),
    (dict(merge_into_out=1), 1),                          # merge mode needs fp32 out
    (dict(merge_into_out=2, out_fp32=1), 1),              # flag is 0 or 1
    (dict(out_final=1 << 24), 1),                         # out_final only in merge mode
    (dict(merge_into_out=1, out_fp32=1, out_final=(1 << 24) + 8), 1),  # misaligned
    (dict(merge_into_out=1, out_fp32=1, out_final=(1 << 20) + 4096), 1),  # overlaps out
    (dict(kv_token_stride=128), 1),                       # below h_kv * d = 256
    (dict(kv_token_stride=260), 1),                       # not a multiple of 8
    (dict(d_v=-1), 1),                                    # negative value head dim
    (dict(d_v=64), 2),                                    # only d = 192 with d_v = 128
    (dict(d=192, d_v=128, kv_token_stride=640), 1),       # packed K/V needs d_v == d
])
def test_fwd_rejects_invalid_arguments_on_host(ga, kw, code):
    p = _params(ga, **kw)
    assert ga.lib().attn_fwd_workspace_bytes(ctypes.byref(p)) == 0
    p.workspace_bytes = 1 << 30
    assert ga.lib().attn_fwd(ctypes.byref(p), None) == code


def test_fwd_accepts_mla_head_dims(ga):
    p = _params(ga, d=192, d_v=128)
    assert ga.lib().attn_fwd_workspace_bytes(ctypes.byref(p)) > 0


def test_binding_workspace_query_takes_v_width(ga):
    """The binding's size query for MLA shapes needs v (its head dim differs
    from k's); without it the shapes read as an unsupported d = 192."""
    import workload
    q, k, v = workload.qkv(1, 256, 4, 2, 192, dv=128)
    ids, pos = workload.segments(1, 256, None)
    assert ga.workspace_bytes_fwd(q, k, ids, pos, v=v) > 0
    assert ga.workspace_bytes_fwd(q, k, ids, pos) == 0
    q, k, v = workload.qkv(1, 256, 4, 2, 128)
    assert ga.workspace_bytes_fwd(q, k, ids, pos, v=v) == ga.workspace_bytes_fwd(q, k, ids, pos)


def test_fwd_workspace_checks(ga):
    p = _params(ga)
    need = ga.lib().attn_fwd_workspace_bytes(ctypes.byref(p))
    assert need > 0
    p.workspace_bytes = need - 1
    assert ga.lib().attn_fwd(ctypes.byref(p), None) == 1
    p.workspace_bytes = need
    p.workspace = (1 << 20) + 128  # not 256-byte aligned
    assert ga.lib().attn_fwd(ctypes.byref(p), None) == 1


def test_bwd_rejects_invalid_arguments_on_host(ga):
    bp = ga.BwdParams()
    bp.fwd = _params(ga)
    assert ga.lib().attn_bwd(ctypes.byref(bp), None) == 1  # dout/dq/dk/dv missing
    bp.dout = bp.dq = bp.dk = bp.dv = 1 << 20
    bp.fwd.out_fp32 = 1
    assert ga.lib().attn_bwd(ctypes.byref(bp), None) == 1
    bp.fwd.out_fp32 = 0
    bp.fwd.merge_into_out = 1
    assert ga.lib().attn_bwd(ctypes.byref(bp), None) == 1
    bp.fwd.merge_into_out = 0
    bp.fwd.workspace_bytes = 1 << 30
    bp.deterministic = 2  # the flag is 0 or 1
    assert ga.lib().attn_bwd(ctypes.byref(bp), None) == 1
    bp.deterministic = 0
    bp.kernel_events[0] = 1 << 12  # timing events come in pairs (never recorded here)
    assert ga.lib().attn_bwd(ctypes.byref(bp), None) == 1
    bp.kernel_events[0] = None
    bp.delta = (1 << 40) + 2  # the optional D output: 4-byte aligned
    assert ga.lib().attn_bwd(ctypes.byref(bp), None) == 1
    bp.delta = bp.fwd.workspace  # ... and clear of the other buffers
    assert ga.lib().attn_bwd(ctypes.byref(bp), None) == 1
    bp.delta = None
    # d = 256 and the MLA shape (192, 128) are taken (by the dK / dV + dQ kernel
    # pair); only the size query runs here, nothing is launched on the fake
    # pointers.  Their workspace holds no fp32 dQ accumulator.
    bp.fwd.d, bp.fwd.kv_token_stride = 256, 0
    n256 = ga.lib().attn_bwd_workspace_bytes(ctypes.byref(bp))
    assert 0 < n256 < 2 * 4096 * 16 * 256 * 4
    bp.fwd.d, bp.fwd.d_v = 192, 128
    assert ga.lib().attn_bwd_workspace_bytes(ctypes.byref(bp)) > 0
    bp.fwd.d_v = 0  # 192 / 192 is no supported shape
    assert ga.lib().attn_bwd_workspace_bytes(ctypes.byref(bp)) == 0
    bp.fwd.d, bp.fwd.d_v = 80, 0
    assert ga.lib().attn_bwd_workspace_bytes(ctypes.byref(bp)) == 0
    # a scale the forward takes but the backward does not: (LSE - ln scale) /
    # scale would leave the fp32 range
    bp.fwd.d = 128
    bp.fwd.scale = 1e-35
    assert ga.lib().attn_bwd(ctypes.byref(bp), None) == 2


@pytest.mark.parametrize("args,code", [
    ((1 << 20, 1 << 20, 1, 64, 16, 0, 4, 1), 1),           # in == out
    ((1 << 20, 1 << 21, 1, 60, 16, 0, 4, 1), 1),           # s % 2R != 0
    ((1 << 20, 1 << 21, 1, 64, 16, 1, 4, 3), 1),           # s % (R*stripe) != 0
    ((1 << 20, 1 << 21, 1, 64, 16, 2, 4, 1), 1),           # unknown strategy
    ((1 << 20, (1 << 20) + 512, 1, 64, 16, 0, 4, 1), 1),   # overlapping buffers
    ((1 << 20, 1 << 21, 1, 64, 16, 0, 0, 1), 1),           # cp_size 0
])
def test_reorder_rejects_invalid_arguments_on_host(ga, args, code):
    assert ga.lib().reorder_causal_lb(*args, None) == code
    assert ga.lib().inverse_reorder_causal_lb(*args, None) == code


def test_merge_rejects_invalid_arguments_on_host(ga):
    a = 1 << 20
    assert ga.lib().attn_merge_partial(None, a, a, a, 0, None, 1, 1, 1, 128, None) == 1
    assert ga.lib().attn_merge_partial(a, a, a, a, 0, None, 1, 1, 1, 12, None) == 1
    assert ga.lib().attn_merge_partial(a + 4, a, a, a, 0, None, 1, 1, 1, 128, None) == 1


def test_device_status_rejects_null(ga):
    assert ga.lib().attn_read_device_status(None, None) == 1


def test_tile_order_rejects_invalid_arguments_on_host(ga):
    """The work-order debug hook validates like attn_tile_plan, before any
    launch (the pointers here are fake and never dereferenced)."""
    p = _params(ga)
    p.workspace_bytes = 1 << 30
    assert ga.lib().attn_tile_order(ctypes.byref(p), None, 1 << 20, None) == 1   # no q_order
    assert ga.lib().attn_tile_order(ctypes.byref(p), 1 << 20, (1 << 20) + 2, None) == 1  # misaligned
    p.workspace_bytes = 16
    assert ga.lib().attn_tile_order(ctypes.byref(p), 1 << 20, 1 << 21, None) == 1  # workspace
    p = _params(ga, d=96)
    assert ga.lib().attn_tile_order(ctypes.byref(p), 1 << 20, 1 << 21, None) == 2  # head dim


def test_segments_rejects_invalid_arguments_on_host(ga):
    a, o = 1 << 20, 1 << 24
    f = ga.lib().attn_segments_from_seqlens
    assert f(None, None, 1, 1, 16, a, o, None) == 1          # no lengths
    assert f(a, None, 1, 0, 16, o, o + (1 << 20), None) == 1  # nseg 0
    assert f(a, None, 1, 1, 0, o, o + (1 << 20), None) == 1   # s 0
    assert f(a + 2, None, 1, 1, 16, o, o + (1 << 20), None) == 1  # misaligned
    assert f(a, None, 1, 8193, 16, o, o + (1 << 20), None) == 2   # too many segments
    assert f(a, None, 1, 1, 16, o, o + 32, None) == 1         # ids / pos overlap
    assert f(a, None, 1, 1, 16, a, o, None) == 1              # ids over the lengths
    assert f(a, o, 1, 4, 16, o + 8, o + (1 << 20), None) == 1   # ids over the offsets
