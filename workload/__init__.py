"""Seeded synthetic workloads for the packed-THD attention hot path.

This module only draws inputs: it holds none of the attention arithmetic, so
both the CPU oracle and the CUDA path may take their inputs from it.

Workload recipe (TransformerEngine JAX tutorial "Context-Parallel Attention",
section 1 "Packed THD inputs"):

* q/k/v (and the output gradient dout) are drawn as float32 N(0, 1) from one
  seeded generator in the order q, k, v, dout, then rounded to bfloat16
  (round-to-nearest-even).  The tutorial seeds its generator with 2026.
* Each batch row is a sequence of ``slots`` equal segment slots.  In a slot of
  length L the first 3L/4 tokens are valid and carry the segment id (1..slots);
  the rest are padding with id 0.  segment_pos restarts at 0 in every slot and
  runs over the padding tokens too.  The same ids/pos are used for every row.
* ``slots=None`` means one unpadded segment: ids all 1, pos 0..s-1.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

SEED = 2026


@dataclass(frozen=True)
class Workload:
    name: str
    b: int
    s: int
    hq: int
    hkv: int
    d: int
    slots: Optional[int]      # None: one segment, no padding
    window_left: int          # -1: unlimited
    bwd: bool = False
    cp_size: int = 0          # >0: ring emulation over cp_size logical shards
    note: str = ""
    d_v: int = 0              # head dim of v / out when it differs from q / k's (0: d)
    fwd_only: bool = False    # measured forward only

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    @property
    def dv(self) -> int:
        return self.d_v or self.d


# The five workloads the hot path is measured and checked on, then the other
# head dims' forward-only shapes.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 256, 4, 2, 64, None, -1,
                     note="one segment, causal, no window"),
    "packed_thd": Workload("packed_thd", 2, 4096, 16, 2, 128, 4, -1,
                           note="4 slots of 1024 (768 valid), causal"),
    "packed_swa": Workload("packed_swa", 2, 16384, 32, 8, 128, 4, 1024, bwd=True,
                           note="4 slots of 4096 (3072 valid), causal, window (1024,0)"),
    "ring_cp4": Workload("ring_cp4", 1, 32768, 64, 8, 128, None, -1, cp_size=4,
                         note="one segment, causal, ring emulation over 4 shards"),
    "full_swa_64k": Workload("full_swa_64k", 2, 65536, 128, 8, 128, 4, 8192, bwd=True,
                             note="4 slots of 16384 (12288 valid), causal, window (8192,0)"),
    # Other head dims (TE tutorial, "next steps": MLA head dims), forward and
    # backward, on the packed_swa packing and on one causal 32k segment.
    "packed_swa_d256": Workload("packed_swa_d256", 2, 16384, 32, 8, 256, 4, 1024, bwd=True,
                                note="packed_swa's packing at d = 256"),
    "packed_swa_mla": Workload("packed_swa_mla", 2, 16384, 32, 8, 192, 4, 1024, d_v=128,
                               bwd=True, note="packed_swa's packing, d_qk 192, d_v 128"),
    "causal_32k_d256": Workload("causal_32k_d256", 1, 32768, 32, 8, 256, None, -1, bwd=True,
                                note="one causal segment of 32768, d = 256"),
    "causal_32k_mla": Workload("causal_32k_mla", 1, 32768, 32, 8, 192, None, -1, d_v=128,
                               bwd=True, note="one causal segment, d_qk 192, d_v 128"),
    # Profiling case: one segment of 32768 with the 64k workload's window and
    # GQA group size, so a query tile meets ~65 key tiles as there, in a
    # problem of a few hundred MB with several waves of CTAs (kernel counters
    # are captured here).
    "swa_32k_g16": Workload("swa_32k_g16", 1, 32768, 32, 2, 128, None, 8192, bwd=True,
                            note="profiling: one segment, window (8192,0), Hq 32, Hkv 2"),
}


def segments(b: int, s: int, slots: Optional[int]):
    """segment_ids, segment_pos as int32 [b, s] (CPU tensors)."""
    if slots is None:
        ids = torch.ones(s, dtype=torch.int32)
        pos = torch.arange(s, dtype=torch.int32)
    else:
        if s % slots:
            raise ValueError("seq must be a multiple of the slot count")
        slot = s // slots
        valid = 3 * slot // 4
        ids_parts, pos_parts = [], []
        for sid in range(1, slots + 1):
            part = torch.zeros(slot, dtype=torch.int32)
            part[:valid] = sid
            ids_parts.append(part)
            pos_parts.append(torch.arange(slot, dtype=torch.int32))
        ids = torch.cat(ids_parts)
        pos = torch.cat(pos_parts)
    return ids[None].repeat(b, 1).contiguous(), pos[None].repeat(b, 1).contiguous()


def qkv(b: int, s: int, hq: int, hkv: int, d: int, *, seed: int = SEED,
        with_dout: bool = False, device="cpu", s_kv: Optional[int] = None,
        dv: Optional[int] = None):
    """bf16 q [b,s,hq,d], k [b,s_kv,hkv,d], v [b,s_kv,hkv,dv] (and dout
    [b,s,hq,dv]), seeded; dv defaults to d.

    Drawn float32 N(0,1) in the order q, k, v, dout and rounded to bf16.
    A CUDA device uses its own seeded generator (values differ from the CPU
    stream, the distribution is the same).
    """
    s_kv = s if s_kv is None else s_kv
    dv = d if dv is None else dv
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def draw(shape):
        return torch.randn(shape, generator=gen, dtype=torch.float32,
                           device=device).to(torch.bfloat16)

    q = draw((b, s, hq, d))
    k = draw((b, s_kv, hkv, d))
    v = draw((b, s_kv, hkv, dv))
    if with_dout:
        return q, k, v, draw((b, s, hq, dv))
    return q, k, v


def make(w: Workload, *, device="cpu", seed: int = SEED, with_dout: Optional[bool] = None):
    """All inputs of a workload: dict of q, k, v, [dout], ids, pos."""
    with_dout = w.bwd if with_dout is None else with_dout
    tensors = qkv(w.b, w.s, w.hq, w.hkv, w.d, seed=seed, with_dout=with_dout, device=device,
                  dv=w.dv)
    ids, pos = segments(w.b, w.s, w.slots)
    out = dict(q=tensors[0], k=tensors[1], v=tensors[2],
               ids=ids.to(device), pos=pos.to(device))
    if with_dout:
        out["dout"] = tensors[3]
    return out


def random_segments(b: int, s: int, *, seed: int, max_segments: int = 4,
                    pad_prob: float = 0.3):
    """Irregular packing for edge-case tests: random segment lengths, random
    padding runs, ids that may repeat across gaps, positions that restart per
    segment.  Returns int32 [b, s] ids and pos."""
    g = torch.Generator().manual_seed(seed)
    ids = torch.zeros(b, s, dtype=torch.int32)
    pos = torch.zeros(b, s, dtype=torch.int32)
    for bi in range(b):
        t = 0
        sid = 0
        while t < s:
            length = int(torch.randint(1, max(2, s // max_segments + 1), (1,), generator=g))
            length = min(length, s - t)
            if float(torch.rand(1, generator=g)) < pad_prob:
                ids[bi, t:t + length] = 0
                pos[bi, t:t + length] = torch.arange(length, dtype=torch.int32)
            else:
                sid += 1
                ids[bi, t:t + length] = sid
                pos[bi, t:t + length] = torch.arange(length, dtype=torch.int32)
            t += length
    return ids, pos
