"""attn_fwd_noalloc: the forward entry point for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).  Called
through the C ABI and compared with attn_fwd (caller-provided workspace) on
two calls in a row, which also checks that the shared scratch left behind by
one call does not disturb the next.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

import workload
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _params(ga, x, w, out, lse):
    p = ga.FwdParams()
    p.q, p.k, p.v = x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr()
    p.q_segment_ids = p.kv_segment_ids = x["ids"].data_ptr()
    p.q_segment_pos = p.kv_segment_pos = x["pos"].data_ptr()
    p.b, p.s_q, p.s_kv, p.h_q, p.h_kv, p.d = w.b, w.s, w.s, w.hq, w.hkv, w.d
    p.window_left, p.window_right, p.scale = w.window_left, 0, w.scale
    p.out_fp32 = 0
    p.out, p.lse = out.data_ptr(), lse.data_ptr()
    p.workspace, p.workspace_bytes = None, 0
    return p


@pytest.mark.parametrize("name", ["packed_swa", "tiny"])
def test_noalloc_matches_attn_fwd_twice(name):
    import long_context_attention_attn_gb300 as ga
    w = workload.WORKLOADS[name]
    x = workload.make(w, device=DEV, with_dout=False)
    ref_o, ref_l = ga.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"],
                               window_left=w.window_left, scale=w.scale)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        p = _params(ga, x, w, out, lse)
        assert ga.lib().attn_fwd_noalloc(ctypes.byref(p), stream) == ga.ATTN_OK
        # the scratch's status word: every bounded device-side wait completed
        assert ga.lib().attn_fwd_noalloc_status(stream) == ga.ATTN_OK
        torch.cuda.synchronize()
        check_out(out.cpu(), ref_o.float().cpu())
        check_lse(lse.cpu(), ref_l.cpu())


def test_noalloc_rejects_oversized_and_invalid_problems():
    import long_context_attention_attn_gb300 as ga
    w = workload.WORKLOADS["tiny"]
    x = workload.make(w, device=DEV, with_dout=False)
    out = torch.empty_like(x["q"])
    lse = torch.empty(w.b, w.hq, w.s, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = _params(ga, x, w, out, lse)
    p.b, p.s_q, p.s_kv = 4, 1 << 20, 1 << 20  # plan would need ~256 MiB of scratch
    assert ga.lib().attn_fwd_noalloc(ctypes.byref(p), stream) == ga.ATTN_ERR_UNSUPPORTED
    p = _params(ga, x, w, out, lse)
    p.window_right = 3
    assert ga.lib().attn_fwd_noalloc(ctypes.byref(p), stream) == ga.ATTN_ERR_INVALID_ARG
