"""GPU parity of the integer / HBM-bound kernels through the C ABI:
reorder + inverse (bit-exact), tile plan (bit-exact), merge (tolerance)."""
import numpy as np
import pytest
import torch

import workload
from oracle import merge as M
from oracle import plan as PL
from oracle import reorder as RO
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ga():
    import long_context_attention_attn_gb300 as pkg
    return pkg


DEV = "cuda"


@pytest.mark.parametrize("shape,seq_dim,dtype,strategy,R,stripe", [
    ((1, 32768, 64, 128), 1, torch.bfloat16, RO.DUAL_CHUNK, 4, 1),   # q of the ring workload
    ((1, 32768, 8, 128), 1, torch.bfloat16, RO.DUAL_CHUNK, 4, 1),    # k / v
    ((1, 32768), 1, torch.int32, RO.DUAL_CHUNK, 4, 1),               # ids / pos
    ((64, 32768), 1, torch.float32, RO.DUAL_CHUNK, 4, 1),            # lse viewed [b*h, s]
    ((2, 4096, 16, 128), 1, torch.bfloat16, RO.STRIPED, 4, 1),
    ((2, 65536, 8, 128), 1, torch.bfloat16, RO.STRIPED, 4, 512),
    ((3, 48, 5), 1, torch.uint8, RO.STRIPED, 3, 2),                  # odd byte rows
    ((2, 40, 3), 1, torch.int32, RO.DUAL_CHUNK, 2, 1),               # 12-byte rows
])
def test_reorder_bit_exact(ga, shape, seq_dim, dtype, strategy, R, stripe):
    g = torch.Generator(device=DEV).manual_seed(7)
    if dtype.is_floating_point:
        x = torch.randn(shape, generator=g, device=DEV).to(dtype)
    else:
        x = torch.randint(0, 120, shape, generator=g, device=DEV).to(dtype)
    y = ga.reorder_causal_lb(x, strategy, R, stripe, seq_dim=seq_dim)
    torch.cuda.synchronize()
    src = torch.from_numpy(RO.src_index(shape[seq_dim], strategy, R, stripe)).to(DEV)
    ref = x.index_select(seq_dim, src)
    assert torch.equal(y.view(torch.uint8) if dtype != torch.uint8 else y,
                       ref.view(torch.uint8) if dtype != torch.uint8 else ref)
    z = ga.inverse_reorder_causal_lb(y, strategy, R, stripe, seq_dim=seq_dim)
    torch.cuda.synchronize()
    assert torch.equal(z, x)


def test_reorder_matches_oracle_on_host_copy(ga):
    x = torch.arange(2 * 24 * 3, dtype=torch.int32).reshape(2, 24, 3)
    y = ga.reorder_causal_lb(x.to(DEV), RO.DUAL_CHUNK, 3).cpu().numpy()
    assert np.array_equal(y, RO.reorder(x.numpy(), RO.DUAL_CHUNK, 3))
    y = ga.reorder_causal_lb(x.to(DEV), RO.STRIPED, 4, 2).cpu().numpy()
    assert np.array_equal(y, RO.reorder(x.numpy(), RO.STRIPED, 4, 2))


def _plan_case(ga, ids, pos, window, s_kv_ids=None, s_kv_pos=None):
    kv_ids = ids if s_kv_ids is None else s_kv_ids
    kv_pos = pos if s_kv_pos is None else s_kv_pos
    b, s = ids.shape
    q = torch.empty(b, s, 2, 64, dtype=torch.bfloat16, device=DEV)
    k = torch.empty(b, kv_ids.shape[1], 1, 64, dtype=torch.bfloat16, device=DEV)
    cls, rng = ga.attn_tile_plan(q, k, ids.to(DEV), pos.to(DEV), kv_ids.to(DEV),
                                 kv_pos.to(DEV), window_left=window)
    torch.cuda.synchronize()
    ref = PL.classes(ids.numpy(), pos.numpy(), kv_ids.numpy(), kv_pos.numpy(), window)
    assert np.array_equal(cls.cpu().numpy(), ref)
    assert np.array_equal(rng.cpu().numpy(), PL.ranges(ref))


@pytest.mark.parametrize("name", ["tiny", "packed_thd", "packed_swa", "ring_cp4", "full_swa_64k"])
def test_plan_bit_exact_on_workloads(ga, name):
    w = workload.WORKLOADS[name]
    ids, pos = workload.segments(w.b, w.s, w.slots)
    if w.s > 20000:  # keep the pure-Python oracle plan within seconds
        ids, pos = ids[:1], pos[:1]
    _plan_case(ga, ids, pos, w.window_left)


# up to 4096 class bytes (b * nq * nk) the plan runs in one CTA, above it as
# the parallel kernels: random packings and cross descriptors on both paths
@pytest.mark.parametrize("seed,s,window", [(1, 1000, -1), (2, 777, 40), (3, 1300, 0),
                                           (4, 9000, -1), (5, 8500, 300), (6, 10000, 0)])
def test_plan_bit_exact_on_random_packing(ga, seed, s, window):
    ids, pos = workload.random_segments(2, s, seed=seed)
    _plan_case(ga, ids, pos, window)


@pytest.mark.parametrize("s,lo,hi", [(1024, 256, 768), (12000, 3000, 9500)])
def test_plan_cross_descriptor(ga, s, lo, hi):
    ids, pos = workload.segments(1, s, None)
    kv_ids, kv_pos = ids[:, lo:hi].contiguous(), pos[:, lo:hi].contiguous()
    _plan_case(ga, ids, pos, 100, kv_ids, kv_pos)


@pytest.mark.parametrize("blk_dtype,final", [(torch.float32, False), (torch.bfloat16, False),
                                             (torch.float32, True)])
def test_merge_matches_oracle(ga, blk_dtype, final):
    b, s, h, d = 2, 1000, 8, 128
    g = torch.Generator().manual_seed(3)
    oa = torch.randn(b, s, h, d, generator=g)
    ob = torch.randn(b, s, h, d, generator=g).to(blk_dtype)
    la = torch.randn(b, h, s, generator=g) * 3
    lb = torch.randn(b, h, s, generator=g) * 3
    la[:, :, :50] = -torch.inf      # accumulator empty
    lb[:, :, 40:90] = -torch.inf    # block empty
    oa[:, :50] = float("nan")       # never read where lse_acc = -inf
    ref_o, ref_l = M.merge_partial(torch.nan_to_num(oa).numpy(), la.numpy(),
                                   ob.float().numpy(), lb.numpy())
    ref_o[:, 40:50] = 0.0
    acc, lacc = oa.to(DEV), la.to(DEV)
    fin = torch.empty(b, s, h, d, dtype=torch.bfloat16, device=DEV) if final else None
    o, l = ga.attn_merge_partial(acc, lacc, ob.to(DEV), lb.to(DEV), out_final=fin)
    torch.cuda.synchronize()
    got = o.float().cpu().numpy()
    check_out(got, ref_o)
    check_lse(l.cpu(), ref_l)
    if not final:
        np.testing.assert_allclose(got, ref_o, atol=1e-5, rtol=1e-5)


@pytest.mark.parametrize("seed", range(4))
def test_segments_from_seqlens_bit_exact(seed):
    """attn_segments_from_seqlens equals the oracle's length -> descriptor map,
    with and without offsets, including empty, negative and cut-off segments."""
    import long_context_attention_attn_gb300 as ga
    from oracle.descriptors import segments_from_seqlens
    rng = np.random.default_rng(seed)
    b, nseg, s = 3, [1, 5, 40, 700][seed], [300, 4097, 9000, 70000][seed]
    lens = rng.integers(-3, max(4, 2 * s // nseg), size=(b, nseg)).astype(np.int32)
    gaps = rng.integers(0, 9, size=(b, nseg))
    offs = (np.cumsum(gaps + np.maximum(lens, 0), axis=1) - np.maximum(lens, 0)).astype(np.int32)
    for offsets in (None, offs):
        want_i, want_p = segments_from_seqlens(lens, s, offsets)
        got_i, got_p = ga.segments_from_seqlens(
            torch.from_numpy(lens).cuda(), s,
            None if offsets is None else torch.from_numpy(offsets).cuda())
        np.testing.assert_array_equal(got_i.cpu().numpy(), want_i)
        np.testing.assert_array_equal(got_p.cpu().numpy(), want_p)


def test_segments_from_seqlens_tutorial_row():
    """The tutorial's padded slots as lengths + offsets reproduce the 64k
    workload's descriptor bit for bit."""
    import long_context_attention_attn_gb300 as ga
    lens = torch.full((2, 4), 12288, dtype=torch.int32, device="cuda")
    offs = torch.tensor([[0, 16384, 32768, 49152]] * 2, dtype=torch.int32, device="cuda")
    ids, pos = ga.segments_from_seqlens(lens, 65536, offs)
    wi, wp = workload.segments(2, 65536, 4)
    assert torch.equal(ids.cpu(), wi) and torch.equal(pos.cpu(), wp)


@pytest.mark.parametrize("det", [False, True])
def test_concurrent_calls_from_host_threads(det):
    """The library keeps no per-call state: four host threads, each with its own
    stream and inputs, calling attn_fwd / attn_bwd at once get bit-identical
    out, lse, dk and dv to the same calls made one after another.  dq is
    compared within the gradient tolerance only: its fp32 sum over key tiles
    is formed by reduce-adds whose order the hardware schedules, so the
    rounding of the last bits may differ from run to run; in deterministic
    mode it is bit-identical too."""
    import threading
    import long_context_attention_attn_gb300 as ga
    cases = []
    for i in range(4):
        q, k, v, dout = workload.qkv(1, 700 + 64 * i, 4, 2, 128 if i % 2 else 64, seed=40 + i,
                                     with_dout=True)
        ids, pos = workload.random_segments(1, 700 + 64 * i, seed=40 + i)
        cases.append(tuple(t.cuda() for t in (q, k, v, dout, ids, pos)))

    def run(c):
        q, k, v, dout, ids, pos = c
        out, lse = ga.attn_fwd(q, k, v, ids, pos, window_left=200, scale=0.1)
        dq, dk, dv = ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, window_left=200, scale=0.1,
                                 deterministic=det)
        return out, lse, dq, dk, dv

    serial = [run(c) for c in cases]
    torch.cuda.synchronize()
    results = [None] * len(cases)

    def worker(i):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(3):
                results[i] = run(cases[i])
        s.synchronize()

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    from tests.parity import check_grad
    for got, want in zip(results, serial):
        out, lse, dq, dk, dv = got
        for name, g, w in (("out", out, want[0]), ("lse", lse, want[1]), ("dk", dk, want[3]),
                           ("dv", dv, want[4])):
            assert torch.equal(g, w), name
        check_grad(dq.cpu(), want[2].cpu(), "dq")
        if det:
            assert torch.equal(dq, want[2])


def _expected_order(w, ctas, sms, reverse):
    """The work order by its rule: heavy first (a stable sort) when the
    heaviest unit's CTA is more than 1/20 of an SM's share of the launch,
    else index order (descending on the query side)."""
    if int(w.max()) * sms * 20 > int(w.sum()) * ctas:
        return np.argsort(-w, kind="stable")
    idx = np.arange(w.size)
    return idx[::-1] if reverse else idx


@pytest.mark.parametrize("name,b,s,hq,hkv,want", [
    # one head: every unit is a large share of the launch, heavy first on both sides
    ("full_swa_64k", None, None, 1, 1, ("sort", "sort")),
    ("packed_thd", None, None, 1, 1, ("sort", "sort")),
    ("ragged", 3, 3000, 1, 1, ("sort", "sort")),        # ragged tail, many equal weights
    # two rows of a million tokens (8192 tiles per row): one causal segment
    # with window 300000 (16384 units, none over 1.1 % of an SM's share:
    # index order), and 3/4 padding then a causal segment of 262144 (weights
    # to 2048, 12288 units of weight 0: heavy first, ties across many chunks)
    ("long_rows", 2, 1 << 20, 1, 1, ("index", "index")),
    ("long_tail_segment", 2, 1 << 20, 1, 1, ("sort", "sort")),
    # the benchmark's workload with its heads: index order on both sides
    ("full_swa_64k", None, None, 128, 8, ("index", "index")),
    # short window, few units: heavy first on both sides
    ("packed_swa", None, None, 32, 8, ("sort", "sort")),
    # one causal segment: index order for the queries, heavy first for the keys
    ("ring_cp4", None, None, 64, 8, ("index", "sort")),
])
def test_work_order_follows_its_rule(name, b, s, hq, hkv, want):
    """The kernels' work order equals the rule's order computed on the host
    from the plan weights (bit for bit, both sides): a stable heaviest-first
    argsort, or index order, as the tail ratio decides; at the 64k workload
    with one head and with its 128 / 8 heads, and at two rows of a million
    tokens in both orders (no cap on the weights)."""
    import long_context_attention_attn_gb300 as ga
    if name in workload.WORKLOADS:
        w = workload.WORKLOADS[name]
        b, s, slots, window = w.b, w.s, w.slots, w.window_left
        ids, pos = workload.segments(b, s, slots)
    elif name == "long_rows":
        ids, pos = workload.segments(b, s, None)  # one causal segment per row
        window = 300000
    elif name == "long_tail_segment":
        ids = torch.zeros(b, s, dtype=torch.int32)
        pos = torch.zeros(b, s, dtype=torch.int32)
        ids[:, 3 * s // 4:] = 1
        pos[:, 3 * s // 4:] = torch.arange(s // 4, dtype=torch.int32)
        window = -1
    else:
        ids, pos = workload.random_segments(b, s, seed=3)
        window = 700
    dev_ids, dev_pos = ids.cuda(), pos.cuda()
    # only shapes are read
    q = torch.empty(b, s, hq, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(b, s, hkv, 64, dtype=torch.bfloat16, device="cuda")
    cls, _ = ga.attn_tile_plan(q, k, dev_ids, dev_pos, window_left=window)
    qo, ko = ga.attn_tile_order(q, k, dev_ids, dev_pos, window_left=window)
    torch.cuda.synchronize()
    del q, k
    c = cls.cpu().numpy() != 0
    q_w = c.sum(axis=2).reshape(-1)
    k_w = c.sum(axis=1).reshape(-1)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    q_ctas = hkv * -(-(hq // hkv) // 2)  # forward: one CTA per kv head and pair of query heads
    k_ctas = hkv                         # fused backward: one CTA per kv head
    eq = _expected_order(q_w, q_ctas, sms, True)
    ek = _expected_order(k_w, k_ctas, sms, False)
    np.testing.assert_array_equal(qo.cpu().numpy(), eq)
    np.testing.assert_array_equal(ko.cpu().numpy(), ek)
    # the case covers the branch it is listed for (on one causal segment the
    # key side's sort is the index order itself: weights fall with the index)
    rule = lambda w, ctas: "sort" if int(w.max()) * sms * 20 > int(w.sum()) * ctas else "index"
    assert (rule(q_w, q_ctas), rule(k_w, k_ctas)) == want


@pytest.mark.parametrize("det", [False, True])
def test_bwd_kernel_events_bracket_the_main_kernel(ga, det):
    """attn_bwd's timing hook: the two events it records around its main
    kernel(s) give a positive time inside the whole call's, and the gradients
    are those of a call without the hook (bit for bit where the path is
    deterministic; dK / dV always)."""
    w = workload.WORKLOADS["packed_swa"]
    x = workload.make(w, device=DEV, with_dout=True)
    q, k, v, ids, pos, dout = x["q"], x["k"], x["v"], x["ids"], x["pos"], x["dout"]
    out, lse = ga.attn_fwd(q, k, v, ids, pos, window_left=w.window_left, scale=w.scale)
    kw = dict(window_left=w.window_left, scale=w.scale, deterministic=det)
    ref = ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, **kw)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record()
    got = ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, kernel_events=(ev[1], ev[2]), **kw,
                      check_status=True)
    ev[3].record()
    torch.cuda.synchronize()
    kernel_ms, call_ms = ev[1].elapsed_time(ev[2]), ev[0].elapsed_time(ev[3])
    assert 0 < kernel_ms < call_ms
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    if det:
        assert torch.equal(got[0], ref[0])


@pytest.mark.parametrize("name", ["tiny", "packed_thd"])
def test_fwd_bwd_replay_from_cuda_graph(ga, name):
    """A whole fwd + bwd step captured once in a CUDA graph (every call only
    enqueues work on the stream; the tensor maps are kernel arguments by
    value) and replayed on new inputs written in place gives what eager calls
    give on those inputs: forward bit for bit, dK / dV bit for bit, dQ bit for
    bit in the deterministic mode."""
    w = workload.WORKLOADS[name]
    x = workload.make(w, device=DEV, with_dout=True)
    q, k, v, ids, pos, dout = x["q"], x["k"], x["v"], x["ids"], x["pos"], x["dout"]
    kw = dict(window_left=w.window_left, scale=w.scale)
    wsf = torch.empty(ga.workspace_bytes_fwd(q, k, ids, pos, **kw, v=v), dtype=torch.uint8,
                      device=DEV)
    wsb = torch.empty(ga.workspace_bytes_bwd(q, k, ids, pos, w.window_left, v=v,
                                             deterministic=True), dtype=torch.uint8, device=DEV)
    out, lse = torch.empty_like(q), torch.empty(w.b, w.hq, w.s, dtype=torch.float32, device=DEV)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step():
        ga.attn_fwd(q, k, v, ids, pos, out=out, lse=lse, workspace=wsf, **kw)
        ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, dq=dq, dk=dk, dv=dv, workspace=wsb,
                    deterministic=True, **kw)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside the capture (kernel attributes set once)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    y = workload.make(w, device=DEV, with_dout=True, seed=workload.SEED + 7)
    for name_, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        t.copy_(y[name_])
    g.replay()
    torch.cuda.synchronize()
    got = [t.clone() for t in (out, lse, dq, dk, dv)]
    assert ga.read_device_status(wsf) == 0 and ga.read_device_status(wsb) == 0
    ro, rl = ga.attn_fwd(q, k, v, ids, pos, **kw)
    rq, rk, rv = ga.attn_bwd(q, k, v, ro, rl, dout, ids, pos, deterministic=True, **kw)
    torch.cuda.synchronize()
    for a_, b_ in zip(got, (ro, rl, rq, rk, rv)):
        assert torch.equal(a_, b_)
