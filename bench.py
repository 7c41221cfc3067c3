"""Benchmark: packed-THD GQA sliding-window attention, forward + backward.

One step = attn_fwd + attn_bwd (tile plan, fused forward, D pre-pass, fused
backward, dQ finalise: every row of the hot path that a training step runs)
on the 64k packed workload of the TE tutorial: b=2, s=65536 (4 slots of 16384
with 12288 valid tokens), 128 query heads, 8 kv heads, d=128, causal with a
(8192, 0) window, bf16.  Throughput counts valid (query, key) pairs only:
4*d FLOP per pair and head forward, 10*d backward (S recomputed).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs its own independent
instance of the workload (weak scaling, no data-path collective); the step
time is the maximum over ranks.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload (rank 0 only).

The JSON line also carries: `roofline` for the backward kernel alone (timed
between CUDA events attn_bwd records around its launch; `roofline.call` has
the whole call), `e2e` (every step's inputs copied in from pinned host memory
and its loss vdot(out, dout) read back) and `e2e_grads_out` (dq, dk, dv copied
back instead), `cpu_baseline` (the oracle on the host cores), `clocks`
(nvidia-smi during the timed region) and `components.per_config` (every
workload of the pages' set, the ring and all-gather emulations, the
deterministic backward, CUDA-graph replays of the small steps).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s on valid pairs, % of GB300 dense BF16 peak (1 GPU)"
METRIC_FWD = "attention fwd TFLOP/s on valid pairs, % of GB300 dense BF16 peak (1 GPU)"
WORKLOAD = "full_swa_64k"
# TE tutorial, section 5: single-GPU fused attention fwd+bwd on this exact
# workload, 126.687 ms on one GB200 (context, another machine).
PAGE_GB200_MS = 126.68747901916504


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload fwd / bwd, ring and all-gather timings")
    ap.add_argument("--deterministic", action="store_true",
                    help="time attn_bwd(deterministic=True): the dK / dV + dQ kernel pair")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload name (the headline number is full_swa_64k; smaller ones "
                         "serve profiling)")
    return ap.parse_args()


def median(xs):
    xs = sorted(xs)
    n = len(xs)
    return xs[n // 2] if n % 2 else 0.5 * (xs[n // 2 - 1] + xs[n // 2])


def max_over_ranks(value, dist=None, device="cpu"):
    """The slowest rank's figure (every rank calls this with its own)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flop_per_rank_step, ms_per_step):
    """Whole-job throughput: every rank runs one instance per step (weak
    scaling), timed by the slowest rank."""
    return world * flop_per_rank_step / (ms_per_step * 1e-3) / 1e12


def valid_pairs(w):
    """Exact visible-pair count of the workload (per head, all batch rows),
    counted from the segment descriptor: per segment of L valid tokens with an
    inclusive window W, sum over positions p of min(p, W) + 1."""
    import workload
    ids, pos = workload.segments(w.b, w.s, w.slots)
    total = 0
    for bi in range(w.b):
        i, p = ids[bi].tolist(), pos[bi].tolist()
        seg_len = {}
        for sid in i:
            if sid:
                seg_len[sid] = seg_len.get(sid, 0) + 1
        for sid, L in seg_len.items():
            W = w.window_left
            if W < 0 or W >= L - 1:
                total += L * (L + 1) // 2
            else:
                total += (W + 1) * (W + 2) // 2 + (L - W - 1) * (W + 1)
    return total


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return dict(bf16_burst=m["bf16_tflops"], bf16_sustained=m["bf16_tflops_sustained"],
                    hbm_gbs=m["hbm_gbs"], source="measured (MEASURED_PEAKS.json)")
    return dict(bf16_burst=1900.0, bf16_sustained=1700.0, hbm_gbs=6800.0,
                source="fallback (profiling recipe)")


def bwd_traffic():
    """DRAM bytes per launch of the fused backward kernel on the benchmark
    workload, from the committed ncu summary, or None once the kernel sources
    (the kernel itself and the plan that orders its work) differ from the
    ones that summary was taken with."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "attn_bwd_dram_full_swa_64k.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.split(":")[0] in ("dram_bytes_read_per_launch",
                                                   "dram_bytes_write_per_launch",
                                                   "source_sha256"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    csrc = os.path.join(ROOT, "long_context_attention_attn_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("attn_bwd.cu", "kernels_misc.cu", "ptx.cuh", "internal.h"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    if vals.get("source_sha256") != h.hexdigest():
        return None
    return int(vals["dram_bytes_read_per_launch"]) + int(vals["dram_bytes_write_per_launch"])


class Clocks:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # raw samples (the JSON line carries the summary); BENCH_CLOCKS_DIR keeps them
        out_dir = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_rank{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["no samples"]}
        loaded = sorted(sm)[len(sm) // 4:] or sm  # drop idle ramp samples
        med = sorted(loaded)[len(loaded) // 2]
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_sample(w, budget_s=12.0, max_blocks=48):
    """Times the CPU oracle (fwd + bwd) on query-row blocks of one kv group of
    the workload until ~budget_s seconds of CPU work; returns (TFLOP/s, info)."""
    import numpy as np
    import torch

    import workload
    from oracle import attention as A

    torch.set_num_threads(os.cpu_count() or 1)
    g = w.hq // w.hkv
    # Sample: batch row 0, kv group 0 (all its query heads), query-row blocks of
    # 64 from position 9000 of the first segment (window fully open).  The
    # inputs are cut to the first segment's valid tokens, which hold every key
    # those rows can see; positions travel with the tokens.
    n_tok = 3 * (w.s // w.slots) // 4 if w.slots else w.s
    ids, pos = workload.segments(1, w.s, w.slots)
    ids, pos = ids[:, :n_tok].numpy(), pos[:, :n_tok].numpy()
    q, k, v, dout = (t[:, :n_tok].to(torch.float64).numpy() for t in
                     workload.qkv(1, w.s, g, 1, w.d, seed=workload.SEED, with_dout=True,
                                  dv=w.dv))
    flops = 0.0
    t0 = time.perf_counter()
    blocks = 0
    r0 = min(9000, n_tok - 64 * max_blocks)
    while blocks < max_blocks:
        rows = np.arange(r0 + 64 * blocks, r0 + 64 * (blocks + 1))
        A.attn_fwd(q, k, v, ids, pos, ids, pos, w.window_left, w.scale, rows=rows)
        A.attn_bwd(q, k, v, dout, ids, pos, ids, pos, w.window_left, w.scale, rows=rows)
        W = w.window_left
        pairs = sum((int(p) if W < 0 else min(int(p), W)) + 1 for p in pos[0, rows])
        flops += pairs * g * (8 * w.d + 6 * w.dv)  # fwd 2 (d + d_v) + bwd 2 (3 d + 2 d_v)
        blocks += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    info = dict(cores=torch.get_num_threads(),
                sample=f"{blocks} blocks of 64 query rows from position {r0} x {g} heads (kv group 0, "
                       f"batch 0) of {w.name}, fwd+bwd, {dt:.1f} s")
    return flops / dt / 1e12, info


def host_link(h, d, h_back, stream):
    """Pinned host <-> device copy bandwidth of this machine (GB/s), measured with
    CUDA events on the copy stream: the bound of the end-to-end figure, whose
    step moves its inputs in and its gradients out."""
    import torch
    res = {}
    for name, dst, src in (("h2d_gbs", d, h), ("d2h_gbs", h_back, d)):
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)  # warm-up
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(3):
                dst.copy_(src, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        res[name] = 3 * src.numel() * src.element_size() / (e0.elapsed_time(e1) * 1e-3) / 1e9
    # both directions at once (the end-to-end step overlaps them; the copied
    # contents are not used): on these boxes the sum is below the two one-way
    # figures added together
    s2 = torch.cuda.Stream(device=stream.device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    s2.wait_event(e0)
    with torch.cuda.stream(stream):
        for _ in range(3):
            d.copy_(h, non_blocking=True)
    with torch.cuda.stream(s2):
        for _ in range(3):
            h_back.copy_(d, non_blocking=True)
    stream.wait_stream(s2)
    e1.record(stream)
    torch.cuda.synchronize()
    nb = h.numel() * h.element_size()
    res["both_gbs"] = 3 * (nb + h_back.numel() * h_back.element_size()) / (e0.elapsed_time(e1) * 1e-3) / 1e9
    res["bytes"] = nb
    return res


def hbm_components(ga, dev, pk):
    """HBM-bound rows of the hot path at the ring workload's shapes (b=1,
    s=32768, 64 query heads, d=128): one merge of a full-sequence fp32 partial
    into an fp32 accumulator (12*d+12 bytes per row-head), and the dual-chunk
    reorder of q (2 x 1 GiB).  CUDA events around 10 back-to-back calls after 3
    warm-ups (so the host's per-call launch latency overlaps the previous call
    instead of counting as kernel time), per call."""
    import torch

    b, s, h, d = 1, 32768, 64, 128
    g = torch.Generator(device=dev).manual_seed(5)
    acc = torch.randn(b, s, h, d, generator=g, device=dev)
    blk = torch.randn(b, s, h, d, generator=g, device=dev)
    la = torch.randn(b, h, s, generator=g, device=dev)
    lb = torch.randn(b, h, s, generator=g, device=dev)
    q = torch.randn(b, s, h, d, generator=g, device=dev).to(torch.bfloat16)
    qo = torch.empty_like(q)

    def timed(fn, n=10):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    merge_ms = timed(lambda: ga.attn_merge_partial(acc, la, blk, lb))
    merge_bytes = b * s * h * (12 * d + 12)
    reorder_ms = timed(lambda: ga.reorder_causal_lb(q, ga.DUAL_CHUNK, 4, out=qo))
    reorder_bytes = 2 * q.numel() * q.element_size()
    out = {"merge_gbs": merge_bytes / (merge_ms * 1e-3) / 1e9,
           "merge_bytes": merge_bytes, "merge_ms": merge_ms,
           "reorder_gbs": reorder_bytes / (reorder_ms * 1e-3) / 1e9,
           "reorder_bytes": reorder_bytes, "reorder_ms": reorder_ms}
    out["merge_pct_hbm"] = 100 * out["merge_gbs"] / pk["hbm_gbs"]
    out["reorder_pct_hbm"] = 100 * out["reorder_gbs"] / pk["hbm_gbs"]
    del acc, blk, la, lb, q, qo
    torch.cuda.empty_cache()
    return out


def _timed_calls(fn, iters=10, warmup=3):
    """Median CUDA-event time (ms) of single calls of fn on the current stream."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return median(times)


def per_config(ga, dev, pk, big=None):
    """fwd / bwd TFLOP/s (valid pairs; medians of 10 single calls after 3
    warm-ups) on every workload of the pages' set, the ring workload as one
    call, as R = 4 logical ring shards (fused and separate merge, forward and
    backward), and the all-gather strategy (forward and backward) at the
    tutorial's 64k shape with stripe 512 (``big`` = the resident full_swa_64k
    inputs, if any)."""
    import torch

    import workload
    from long_context_attention_attn_gb300 import ring

    res = {}
    for name in ("tiny", "packed_thd", "packed_swa", "ring_cp4"):
        w = workload.WORKLOADS[name]
        pairs = valid_pairs(w)
        x = workload.make(w, device=dev, with_dout=True)
        q, k, v, ids, pos, dout = x["q"], x["k"], x["v"], x["ids"], x["pos"], x["dout"]
        ws = torch.empty(ga.workspace_bytes_bwd(q, k, ids, pos, w.window_left),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
        lse = torch.empty(w.b, w.hq, w.s, dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        fwd = lambda: ga.attn_fwd(q, k, v, ids, pos, window_left=w.window_left, scale=w.scale,
                                  out=out, lse=lse, workspace=ws)
        bwd = lambda: ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, window_left=w.window_left,
                                  scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=ws)
        f_ms = _timed_calls(fwd)
        b_ms = _timed_calls(bwd)
        if ga.read_device_status(ws) != 0:
            raise RuntimeError(f"{name}: device status {ga.read_device_status(ws)}")
        ff, bf = 4 * w.d * w.hq * pairs, 10 * w.d * w.hq * pairs
        res[name] = {"fwd_ms": f_ms, "bwd_ms": b_ms, "fwd_tflops": ff / f_ms / 1e9,
                     "bwd_tflops": bf / b_ms / 1e9, "step_tflops": (ff + bf) / (f_ms + b_ms) / 1e9,
                     "valid_pairs_per_head": pairs}
        if name != "ring_cp4":
            # the same fwd + bwd step captured once in a CUDA graph and replayed:
            # the small workloads are bound by their ~20 launches per step
            def both():
                fwd()
                bwd()
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                both()
            torch.cuda.current_stream(dev).wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                both()
            g_ms = _timed_calls(graph.replay)
            if ga.read_device_status(ws) != 0:
                raise RuntimeError(f"{name} (graph): device status {ga.read_device_status(ws)}")
            res[name]["step_graph_ms"] = g_ms
            res[name]["step_graph_tflops"] = (ff + bf) / g_ms / 1e9
            del graph
        if name == "ring_cp4":
            R = w.cp_size
            kw = dict(window_left=w.window_left, scale=w.scale, check_status=False)
            rf = lambda: ring.ring_attn_fwd(q, k, v, ids, pos, R, fused_merge=True, **kw)
            rs = lambda: ring.ring_attn_fwd(q, k, v, ids, pos, R, fused_merge=False, **kw)
            rb = lambda: ring.ring_attn_bwd(q, k, v, out, lse, dout, ids, pos, R, **kw)
            bf_ = lambda: ring.ring_attn_fwd(q, k, v, ids, pos, R, fused_merge=True,
                                             batch_shards=True, **kw)
            bb_ = lambda: ring.ring_attn_bwd(q, k, v, out, lse, dout, ids, pos, R,
                                             batch_shards=True, **kw)
            fused_ms, sep_ms, rb_ms = _timed_calls(rf), _timed_calls(rs), _timed_calls(rb)
            bfw_ms, bbw_ms = _timed_calls(bf_), _timed_calls(bb_)
            res["ring_cp4_shards"] = {
                "what": f"{R} logical dual-chunk ring shards: reorder, {R}x{R} block attn_fwd "
                        "calls with the merge folded into the epilogue (fused) or as a separate "
                        "attn_merge_partial pass, inverse reorder; backward: per-block attn_bwd "
                        "in fp32 accumulate mode with the final LSE",
                "fwd_fused_ms": fused_ms, "fwd_separate_ms": sep_ms, "bwd_ms": rb_ms,
                "fwd_fused_tflops": ff / fused_ms / 1e9, "fwd_separate_tflops": ff / sep_ms / 1e9,
                "bwd_tflops": bf / rb_ms / 1e9,
                "batched": {"what": "batch_shards=True: one call per ring step over all "
                                    "shards, the held K/V blocks (and dK / dV sums) rotated "
                                    "between steps",
                            "fwd_ms": bfw_ms, "bwd_ms": bbw_ms,
                            "fwd_tflops": ff / bfw_ms / 1e9, "bwd_tflops": bf / bbw_ms / 1e9}}
        del x, q, k, v, ids, pos, dout, ws, out, lse, dq, dk, dv
        torch.cuda.empty_cache()
    if big is not None:
        w = workload.WORKLOADS["full_swa_64k"]
        pairs = valid_pairs(w)
        # the deterministic backward (dK / dV kernel + dQ kernel) on the same inputs
        q, k, v, ids, pos = big["q"], big["k"], big["v"], big["ids"], big["pos"]
        out = torch.empty_like(q)
        lse = torch.empty(w.b, w.hq, w.s, dtype=torch.float32, device=dev)
        ws = torch.empty(ga.workspace_bytes_bwd(q, k, ids, pos, w.window_left, deterministic=True),
                         dtype=torch.uint8, device=dev)
        ga.attn_fwd(q, k, v, ids, pos, window_left=w.window_left, scale=w.scale, out=out,
                    lse=lse, workspace=ws)
        grads = [torch.empty_like(t) for t in (q, k, v)]
        det = lambda: ga.attn_bwd(q, k, v, out, lse, big["dout"], ids, pos,
                                  window_left=w.window_left, scale=w.scale, dq=grads[0],
                                  dk=grads[1], dv=grads[2], workspace=ws, deterministic=True)
        det_ms = _timed_calls(det, iters=5)
        if ga.read_device_status(ws) != 0:
            raise RuntimeError("deterministic backward: device status")
        res["full_swa_64k_deterministic_bwd"] = {
            "what": "attn_bwd(deterministic=True): dK / dV kernel + dQ kernel, dQ summed on "
                    "chip in a fixed order (bit-identical run to run)",
            "bwd_ms": det_ms, "bwd_tflops": 10 * w.d * w.hq * pairs / det_ms / 1e9}
        del ws, grads
        torch.cuda.empty_cache()
        ag = lambda: ring.allgather_attn_fwd(q, k, v, ids, pos, 4, window_left=w.window_left,
                                             scale=w.scale, stripe_size=512, check_status=False)
        agb = lambda: ring.allgather_attn_bwd(q, k, v, out, lse, big["dout"], ids, pos, 4,
                                              window_left=w.window_left, scale=w.scale,
                                              stripe_size=512, check_status=False)
        ag_ms = _timed_calls(ag, iters=5)
        agb_ms = _timed_calls(agb, iters=5)
        ff, bf = 4 * w.d * w.hq * pairs, 10 * w.d * w.hq * pairs
        res["allgather_64k"] = {
            "what": "full_swa_64k as 4 logical all-gather shards (striped reorder, stripe 512; "
                    "forward: each shard's queries against the whole reordered K/V in one "
                    "attn_fwd; backward: one attn_bwd per shard against the whole K/V, dK / dV "
                    "accumulated over the shards in fp32; inverse reorder)",
            "fwd_ms": ag_ms, "fwd_tflops": ff / ag_ms / 1e9, "bwd_ms": agb_ms,
            "bwd_tflops": bf / agb_ms / 1e9, "step_tflops": (ff + bf) / (ag_ms + agb_ms) / 1e9}
        del out, lse
        torch.cuda.empty_cache()
    return res


def run_reference(args, rank):
    import workload
    w = workload.WORKLOADS[args.workload]
    if rank != 0:
        return
    vals = []
    info = None
    for i in range(args.warmup + args.steps):
        val, info = oracle_sample(w, budget_s=2.0, max_blocks=2)
        if i >= args.warmup:
            vals.append(val)
    value = sum(vals) / len(vals)
    pairs = valid_pairs(w)
    flops = pairs * w.hq * (8 * w.d + 6 * w.dv)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": flops / (value * 1e12) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "b": w.b, "s": w.s, "hq": w.hq, "hkv": w.hkv, "d": w.d,
                   "window": [w.window_left, 0], "step": "fwd+bwd (CPU oracle, sampled rows)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": info["cores"],
                         "kind": "oracle", "sample": info["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def plan_launches(w):
    """Kernels one attn_fwd and one attn_bwd call launch on this workload.

    The tile plan is one kernel when b * ceil(s/128)^2 <= 4096 (and each side
    has at most 1024 tiles), else two summaries, the classes and four order
    kernels per side, plus the key ranges on the backward.  Forward: plan +
    fused kernel; backward: plan + D pre-pass + fused kernel + dQ finalise, or
    + dK / dV kernel + dQ kernel (same count)."""
    nq = -(-w.s // 128)
    small = w.b * nq <= 1024 and w.b * nq * nq <= 4096
    fwd = (1 if small else 7) + 1
    bwd = (1 if small else 12) + 3
    return fwd, bwd


def run_ours(args, rank, world, local_rank):
    import torch

    import long_context_attention_attn_gb300 as ga
    import workload
    from long_context_attention_attn_gb300 import _build

    if not os.path.exists(ga.LIB_PATH):
        _build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = workload.WORKLOADS[args.workload]
    fwd_only = w.fwd_only  # a forward-only workload: the step is attn_fwd
    pairs = valid_pairs(w)
    fwd_flop = 2 * (w.d + w.dv) * w.hq * pairs
    # backward per pair and head: S and dK, dQ over d_qk; dP and dV over d_v
    bwd_flop = 0 if fwd_only else 2 * (3 * w.d + 2 * w.dv) * w.hq * pairs
    x = workload.make(w, device=dev, with_dout=not fwd_only, seed=workload.SEED + rank)
    q, k, v, ids, pos = x["q"], x["k"], x["v"], x["ids"], x["pos"]
    dout = x.get("dout")
    out = torch.empty(w.b, w.s, w.hq, w.dv, dtype=q.dtype, device=dev)
    lse = torch.empty(w.b, w.hq, w.s, dtype=torch.float32, device=dev)
    if fwd_only:
        ws = torch.empty(ga.workspace_bytes_fwd(q, k, ids, pos, window_left=w.window_left, v=v),
                         dtype=torch.uint8, device=dev)
    else:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(ga.workspace_bytes_bwd(q, k, ids, pos, w.window_left, v=v,
                                                deterministic=args.deterministic),
                         dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        ga.attn_fwd(q, k, v, ids, pos, window_left=w.window_left, scale=w.scale, out=out,
                    lse=lse, workspace=ws)
        if ev:
            ev[1].record(stream)
        if not fwd_only:
            # ev[3] / ev[4]: recorded by attn_bwd right before and after its main
            # kernel(s), the roofline's timing
            ga.attn_bwd(q, k, v, out, lse, dout, ids, pos, window_left=w.window_left,
                        scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                        deterministic=args.deterministic,
                        kernel_events=(ev[3], ev[4]) if ev else None)
        if ev:
            ev[2].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    status = ga.read_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {ga.status_string(status)}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = Clocks(local_rank)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with clocks:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    # per-call figures: medians over the timed steps
    fwd_avg = median([e[0].elapsed_time(e[1]) for e in evs])
    bwd_avg = median([e[1].elapsed_time(e[2]) for e in evs])
    bwd_kernel_ms = None if fwd_only else median([e[3].elapsed_time(e[4]) for e in evs])
    ms_per_step = max_over_ranks(total_ms / args.steps, dist, dev)
    value = whole_job_tflops(world, fwd_flop + bwd_flop, ms_per_step)

    # End to end through the public API, every step: the step's inputs copied
    # host -> device from pinned memory and the step's result read back.  The
    # result is the loss vdot(out, dout) whose gradient the step computes (the
    # sum of the D vector attn_bwd returns in `delta`; the gradients stay on
    # the device, as an optimizer would use them there): `e2e`.  With every
    # gradient copied back to the host instead: `e2e_grads_out`.  As in a
    # training loop with prefetch, the copies run on a copy stream of their own
    # into double-buffered device tensors, so step i+1's inputs (and step
    # i-1's results) move while step i computes; one copy at a time, since on
    # some of these boxes the link moves far less with both directions at once
    # than with either alone (host_link.both_gbs).
    e2e = e2e_grads = None
    if not args.no_e2e and not fwd_only:
        h_in = {n: t.cpu().pin_memory() for n, t in (("q", q), ("k", k), ("v", v),
                                                         ("dout", dout), ("ids", ids),
                                                         ("pos", pos))}
        h_out = [{n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                  for n, t in (("dq", dq), ("dk", dk), ("dv", dv))} for _ in range(2)]
        h_loss = [torch.empty(1, dtype=torch.float32, pin_memory=True) for _ in range(2)]
        d_in = [{n: torch.empty_like(t, device=dev) for n, t in h_in.items()} for _ in range(2)]
        d_out = [(dq, dk, dv), (torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv))]
        delta = [torch.empty(w.b, w.hq, w.s, dtype=torch.float32, device=dev) for _ in range(2)]
        loss = [torch.empty(1, dtype=torch.float32, device=dev) for _ in range(2)]
        bi = sum(t.numel() * t.element_size() for t in h_in.values())
        s_copy = torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()
        h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        fwd_in_done = [ev(), ev()]  # q, k, v, ids, pos of the set have landed (dout may not)
        for e_ in comp_done + d2h_done:
            e_.record(stream)

        def h2d(i):
            sl = i % 2
            s_copy.wait_event(comp_done[sl])  # step i-2 no longer reads this input set
            with torch.cuda.stream(s_copy):
                # the forward's inputs first; dout (read by the backward only) last
                for n in ("q", "k", "v", "ids", "pos", "dout"):
                    d_in[sl][n].copy_(h_in[n], non_blocking=True)
                    if n == "pos":
                        fwd_in_done[sl].record(s_copy)
            h2d_done[sl].record(s_copy)

        def compute(i, grads_out):
            sl = i % 2
            stream.wait_event(fwd_in_done[sl])
            stream.wait_event(d2h_done[sl])  # step i-2's results have left this set
            x_ = d_in[sl]
            gq, gk, gv = d_out[sl]
            ga.attn_fwd(x_["q"], x_["k"], x_["v"], x_["ids"], x_["pos"],
                        window_left=w.window_left, scale=w.scale, out=out, lse=lse, workspace=ws)
            stream.wait_event(h2d_done[sl])  # dout, for the backward
            ga.attn_bwd(x_["q"], x_["k"], x_["v"], out, lse, x_["dout"], x_["ids"], x_["pos"],
                        window_left=w.window_left, scale=w.scale, dq=gq, dk=gk, dv=gv,
                        workspace=ws, deterministic=args.deterministic,
                        delta=None if grads_out else delta[sl])
            if not grads_out:
                torch.sum(delta[sl].view(-1), 0, keepdim=True, out=loss[sl])
            comp_done[sl].record(stream)

        def d2h(i, grads_out):
            sl = i % 2
            s_copy.wait_event(comp_done[sl])
            with torch.cuda.stream(s_copy):
                if grads_out:
                    for n, t in zip(("dq", "dk", "dv"), d_out[sl]):
                        h_out[sl][n].copy_(t, non_blocking=True)
                else:
                    h_loss[sl].copy_(loss[sl], non_blocking=True)
            d2h_done[sl].record(s_copy)

        def run(nsteps, grads_out):
            h2d(0)
            for i in range(nsteps):
                if i + 1 < nsteps:
                    h2d(i + 1)
                compute(i, grads_out)
                d2h(i, grads_out)

        def measure(grads_out):
            run(2, grads_out)
            torch.cuda.synchronize()
            # the same K steps as the device-timed value (the first copy-in and
            # the last copy-out are not hidden behind a neighbouring step), three
            # passes, the median reported: the host link is shared with other
            # tenants on these boxes and can stall one pass
            n_e2e = max(2, args.steps)
            passes = []
            for _ in range(3):
                if dist:
                    dist.barrier()
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s_copy)
                run(n_e2e, grads_out)
                s_copy.wait_stream(stream)
                b_.record(s_copy)
                torch.cuda.synchronize()
                passes.append(max_over_ranks(a.elapsed_time(b_) / n_e2e, dist, dev))
            return median(passes), passes

        link = host_link(h_in["q"], d_in[0]["q"], h_out[0]["dq"], s_copy)
        for grads_out in (False, True):
            e2e_ms, passes = measure(grads_out)
            bo = (sum(t.numel() * t.element_size() for t in h_out[0].values()) if grads_out
                  else h_loss[0].numel() * h_loss[0].element_size())
            rec = {"value": whole_job_tflops(world, fwd_flop + bwd_flop, e2e_ms),
                   "unit": "TFLOP/s", "ms_per_step": e2e_ms, "passes_ms_per_step": passes,
                   "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                   "result": ("dq, dk, dv (bf16)" if grads_out else
                              "the loss vdot(out, dout) = sum of attn_bwd's delta (fp32)"),
                   "copies": "every step's inputs in and its result out inside the timed "
                             "region, on one copy stream (one direction at a time) overlapping "
                             "the neighbouring steps' compute (double-buffered device tensors); "
                             "a step's forward starts once its own inputs have landed, its dout "
                             "copy overlapping it; the median of three passes of the K steps",
                   "host_link": link,
                   # the copies alone, one after the other at the one-way rates
                   "copy_bound_ms": 1e3 * (bi / (link["h2d_gbs"] * 1e9)
                                           + bo / (link["d2h_gbs"] * 1e9))}
            if grads_out:
                e2e_grads = rec
            else:
                e2e = rec
        del h_in, h_out, d_in, d_out, delta

    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return
    pk = peaks()
    fwd_tflops = fwd_flop / (fwd_avg * 1e-3) / 1e12
    if fwd_only:
        print(json.dumps(fwd_only_line(args, w, world, pairs, value, ms_per_step, fwd_avg,
                                       fwd_tflops, pk, clocks)), flush=True)
        return
    hbm = hbm_components(ga, dev, pk)
    per_cfg = None
    if not args.no_per_config:
        per_cfg = per_config(ga, dev, pk, big=x if w.name == WORKLOAD else None)
    bwd_tflops = bwd_flop / (bwd_avg * 1e-3) / 1e12
    bwd_kernel_tflops = bwd_flop / (bwd_kernel_ms * 1e-3) / 1e12
    per_gpu = value / world
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        val, info = oracle_sample(w)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": info["cores"], "kind": "oracle",
               "sample": info["sample"]}
    split_bwd = args.deterministic or w.d == 256 or w.dv != w.d
    fwd_launches, bwd_launches = plan_launches(w)
    launches_per_step = fwd_launches + bwd_launches
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / world / ((fwd_flop + bwd_flop) / (PAGE_GB200_MS * 1e-3) / 1e12),
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "b": w.b, "s": w.s, "slots": w.slots, "hq": w.hq,
                   "hkv": w.hkv, "d": w.d, "d_v": w.dv, "window": [w.window_left, 0],
                   "step": "attn_fwd + attn_bwd" + (" (deterministic)" if args.deterministic
                                                      else ""),
                   "valid_pairs_per_head": pairs,
                   "flop_per_pair_head": {"fwd": 2 * (w.d + w.dv),
                                          "bwd": 2 * (3 * w.d + 2 * w.dv)},
                   "l2": "inputs larger than L2 (q, dout 4 GiB each); no flush",
                   "vs_baseline_ref": "TE tutorial single-GB200 fwd+bwd 126.687 ms on this "
                                      "workload, converted with the same FLOP count",
                   "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU"},
        "pct_of_peak": {"burst": 100 * per_gpu / pk["bf16_burst"],
                        "sustained": 100 * per_gpu / pk["bf16_sustained"],
                        "source": pk["source"]},
        "components": {"fwd_ms": fwd_avg, "bwd_ms": bwd_avg, "fwd_tflops": fwd_tflops,
                       "bwd_tflops": bwd_tflops, "bwd_kernel_ms": bwd_kernel_ms,
                       "bwd_kernel_tflops": bwd_kernel_tflops,
                       "fwd_pct_of_burst_peak": 100 * fwd_tflops / pk["bf16_burst"],
                       "bwd_pct_of_burst_peak": 100 * bwd_tflops / pk["bf16_burst"],
                       "timing": "medians of the timed steps' per-call CUDA events; "
                                 "bwd_kernel_ms: the backward's main kernel(s) alone, between "
                                 "events attn_bwd records around their launch",
                       "hbm_rows": hbm, "per_config": per_cfg},
        "roofline": {"kernel": ("attn_bwd_dkdv_kernel + attn_bwd_dq_tmem_kernel (timed between "
                                "CUDA events attn_bwd records around them, on its stream)"
                                if split_bwd else
                                "attn_bwd_kernel (the fused backward kernel, timed between CUDA "
                                "events attn_bwd records around its launch, on its stream)"),
                     "bound": "tensor", "achieved": bwd_kernel_tflops,
                     "peak": pk["bf16_sustained"], "unit": "TFLOP/s",
                     "frac": bwd_kernel_tflops / pk["bf16_sustained"],
                     "call": {"what": "the whole attn_bwd call (plan, D pre-pass, kernel(s), "
                                      "dQ finalise)", "achieved": bwd_tflops,
                              "frac": bwd_tflops / pk["bf16_sustained"]},
                     "peak_kind": f"bf16 sustained, {pk['source']}",
                     "traffic": bwd_traffic() if (w.name == WORKLOAD and not split_bwd) else None,
                     "traffic_unit": "bytes per launch (ncu dram__bytes_read+write)"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_grads_out": e2e_grads,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def fwd_only_line(args, w, world, pairs, value, ms_per_step, fwd_avg, fwd_tflops, pk, clocks):
    """Result line of a forward-only workload (head dims the backward does not
    take): the step is one attn_fwd call; no end-to-end or oracle leg."""
    per_gpu = value / world
    return {
        "metric": METRIC_FWD, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "b": w.b, "s": w.s, "slots": w.slots, "hq": w.hq,
                   "hkv": w.hkv, "d": w.d, "d_v": w.dv, "window": [w.window_left, 0],
                   "step": "attn_fwd", "valid_pairs_per_head": pairs,
                   "flop_per_pair_head": {"fwd": 2 * (w.d + w.dv)},
                   "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU"},
        "pct_of_peak": {"burst": 100 * per_gpu / pk["bf16_burst"],
                        "sustained": 100 * per_gpu / pk["bf16_sustained"],
                        "source": pk["source"]},
        "components": {"fwd_ms": fwd_avg, "fwd_tflops": fwd_tflops},
        "roofline": {"kernel": "attn_fwd (fused forward + its tile plan; timed per call)",
                     "bound": "tensor", "achieved": fwd_tflops, "peak": pk["bf16_sustained"],
                     "unit": "TFLOP/s", "frac": fwd_tflops / pk["bf16_sustained"],
                     "peak_kind": f"bf16 sustained, {pk['source']}", "traffic": None},
        "cpu_baseline": None,
        "e2e": None,
        "gpu_launches": plan_launches(w)[0] * args.steps,
        "clocks": clocks.summary(),
    }


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
