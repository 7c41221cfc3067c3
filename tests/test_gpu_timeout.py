"""Device-side failure detection without a GPU fault: every wait in the
kernels is bounded.  The test hook withholds all key/value loads, so the
waits run out; the host must then read ATTN_ERR_TIMEOUT from the workspace
status word, and the next normal call must run and be correct."""
import ctypes

import pytest
import torch

import workload
from oracle import attention as A
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_withheld_loads_time_out_and_context_stays_usable():
    import long_context_attention_attn_gb300 as ga
    w = workload.WORKLOADS["tiny"]
    x = workload.make(w)
    g = {k: v.to(DEV) for k, v in x.items()}
    out = torch.empty_like(g["q"])
    lse = torch.empty(w.b, w.hq, w.s, device=DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    p = ga._fwd_params(g["q"], g["k"], g["v"], g["ids"], g["pos"], g["ids"], g["pos"],
                       w.window_left, w.scale, out, lse, False)
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert ga.lib().attn_fwd_test_timeout(ctypes.byref(p), stream) == ga.ATTN_OK
    assert ga.read_device_status(ws) == ga.ATTN_ERR_TIMEOUT
    # the context is still usable: a normal call runs, resets the status and is correct
    o2, l2 = ga.attn_fwd(g["q"], g["k"], g["v"], g["ids"], g["pos"], window_left=w.window_left,
                         scale=w.scale, workspace=ws)
    assert ga.read_device_status(ws) == ga.ATTN_OK
    ro, rl = A.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], x["ids"], x["pos"],
                        w.window_left, w.scale)
    check_out(o2.cpu(), ro)
    check_lse(l2.cpu(), rl)


def test_timeout_raises_through_the_python_api():
    """The bounded-wait timeout reaches a Python caller as AttnError
    (ATTN_ERR_TIMEOUT) when check_status is set, and the next call is sound."""
    import long_context_attention_attn_gb300 as ga
    w = workload.WORKLOADS["tiny"]
    x = workload.make(w)
    g = {k: v.to(DEV) for k, v in x.items()}
    with pytest.raises(ga.AttnError) as ei:
        ga.attn_fwd_test_timeout(g["q"], g["k"], g["v"], g["ids"], g["pos"],
                                 window_left=w.window_left, scale=w.scale)
    assert ei.value.code == ga.ATTN_ERR_TIMEOUT
    out, lse = ga.attn_fwd(g["q"], g["k"], g["v"], g["ids"], g["pos"], window_left=w.window_left,
                           scale=w.scale, check_status=True)
    ro, rl = A.attn_fwd(x["q"], x["k"], x["v"], x["ids"], x["pos"], x["ids"], x["pos"],
                        w.window_left, w.scale)
    check_out(out.cpu(), ro)
    check_lse(lse.cpu(), rl)


def test_ring_driver_raises_when_one_step_times_out(monkeypatch):
    """A ring step whose waits run out makes ring_attn_fwd raise instead of
    returning undefined output: the driver reads every step's status word once
    at the end.  The second attention call of the run is routed to the
    withheld-loads hook (unchecked, like the driver's own calls)."""
    import long_context_attention_attn_gb300 as ga
    from long_context_attention_attn_gb300 import ring
    b, s, hq, hkv, d = 1, 1024, 2, 1, 64
    q, k, v = workload.qkv(b, s, hq, hkv, d, seed=5)
    ids, pos = workload.segments(b, s, None)
    g = [t.to(DEV) for t in (q, k, v, ids, pos)]
    calls = {"n": 0}
    real = ring.attn_fwd

    def flaky(*args, **kw):
        calls["n"] += 1
        if calls["n"] != 2:
            return real(*args, **kw)
        q_, k_, v_, iq, pq, ik, pk = args
        ga.attn_fwd_test_timeout(q_, k_, v_, iq, pq, ik, pk, window_left=kw["window_left"],
                                 scale=kw["scale"], workspace=kw["workspace"],
                                 check_status=False)
        return kw["out"], kw["lse"]

    monkeypatch.setattr(ring, "attn_fwd", flaky)
    with pytest.raises(ga.AttnError) as ei:
        ring.ring_attn_fwd(*g, 2, scale=d ** -0.5, fused_merge=False)
    assert ei.value.code == ga.ATTN_ERR_TIMEOUT
    assert calls["n"] == 4
