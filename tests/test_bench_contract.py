"""CPU checks of bench.py's bookkeeping: the committed DRAM-traffic figure is
used only while the sources it was measured on are unchanged, and the
kernel launch count follows the tile-plan path the library takes (the
threshold read from the CUDA source, so the two cannot drift apart)."""
import hashlib
import re
from pathlib import Path

import bench
import workload

HASHED = ("attn_bwd.cu", "kernels_misc.cu", "ptx.cuh", "internal.h")
ROOT = Path(__file__).resolve().parents[1]


def _fake_tree(tmp_path):
    root = tmp_path / "repo"
    csrc = root / "long_context_attention_attn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in HASHED:
        (csrc / f).write_text(f"// {f}\n")
    h = hashlib.sha256()
    for f in HASHED:
        h.update((csrc / f).read_bytes())
    prof = root / "profiles"
    prof.mkdir()
    (prof / "attn_bwd_dram_full_swa_64k.md").write_text(
        "dram_bytes_read_per_launch: 100\n"
        "dram_bytes_write_per_launch: 23\n"
        f"source_sha256: {h.hexdigest()}\n")
    return root, csrc


def test_traffic_read_only_while_sources_unchanged(tmp_path, monkeypatch):
    root, csrc = _fake_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.bwd_traffic() == 123
    for f in HASHED:  # a change to any hashed source voids the figure
        text = (csrc / f).read_text()
        (csrc / f).write_text(text + "// changed\n")
        assert bench.bwd_traffic() is None
        (csrc / f).write_text(text)
    assert bench.bwd_traffic() == 123


def test_traffic_absent_without_profile(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.bwd_traffic() is None


def test_launch_count_follows_the_plan_threshold():
    src = (ROOT / "long_context_attention_attn_gb300" / "csrc" / "kernels_misc.cu").read_text()
    pairs = int(re.search(r"constexpr int64_t kSmallPlanPairs = (\d+);", src).group(1))
    units = int(re.search(r"constexpr int kSmallPlanUnits = (\d+);", src).group(1))
    nq = int(pairs ** 0.5)
    assert nq * nq == pairs and nq <= units
    base = workload.WORKLOADS["tiny"]

    def shaped(b, s):
        return workload.Workload("t", b, s, base.hq, base.hkv, base.d, None, -1, bwd=True)

    one_cta = (1 + 1, 1 + 3)  # plan kernel + forward; plan + pre-pass + kernel + finalise
    parallel = (7 + 1, 12 + 3)
    assert bench.plan_launches(shaped(1, 128 * nq)) == one_cta           # exactly at the bound
    assert bench.plan_launches(shaped(1, 128 * nq + 1)) == parallel      # one tile more a side
    assert bench.plan_launches(shaped(2, 128 * nq)) == parallel          # twice the class bytes
    assert bench.plan_launches(workload.WORKLOADS["full_swa_64k"]) == parallel
    assert bench.plan_launches(workload.WORKLOADS["tiny"]) == one_cta
