"""Host-side arithmetic of the benchmark (no GPU): the roofline bound and
fraction, the split plan's balance, and the committed traffic lookup keyed by
kernel-source hash."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def test_roofline_hbm_bound():
    # 6 GB at 6000 GB/s = 1 ms; 1 TFLOP at 1800 TF/s = 0.56 ms: HBM binds
    r = bench.roofline_of(6e9, 1e12, 2e-3, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == 3000.0
    assert r["frac"] == 0.5
    assert r["roofline_us"] == 1000.0
    # against the sustained tensor peak: 1 TFLOP / 1400 TF/s = 0.714 ms < 1 ms
    assert r["frac_vs_sustained_tensor_peak"] == 0.5


def test_roofline_tensor_bound_and_sustained():
    # 1.2 GB at 6000 GB/s = 0.2 ms; 0.9 TFLOP at 1800 TF/s = 0.5 ms: tensor binds
    r = bench.roofline_of(1.2e9, 0.9e12, 1e-3, PEAKS)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == 900.0
    assert r["frac"] == 0.5
    assert abs(r["frac_vs_sustained_tensor_peak"] - round(0.9e12 / 1.4e15 / 1e-3, 4)) < 1e-12


def test_plan_balance_matches_brute_force():
    rng = np.random.default_rng(5)
    for _ in range(50):
        seqlens = rng.integers(0, 5000, size=int(rng.integers(1, 200)))
        chunks = int(rng.integers(1, 160))
        granule = int(rng.choice([32, 64, 128]))
        ratio, busy = bench.plan_balance(seqlens, chunks, granule)
        total = int(seqlens.sum())
        if total == 0:
            continue
        # brute force: the smallest multiple of granule (at least one granule)
        # that covers the rows with `chunks` chunks, then each chunk's rows
        cl = granule
        while cl * chunks < total:
            cl += granule
        rows = []
        start = 0
        while start < total:
            rows.append(min(cl, total - start))
            start += cl
        assert busy == len(rows)
        assert abs(ratio - round(max(rows) / (sum(rows) / len(rows)), 4)) < 1e-12


def test_committed_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    rec = {"kernel": "k", "source_hash": "abc123", "dram_bytes_per_launch": 42}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "t.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("abc123", "t.json") == 42
    assert bench.committed_traffic("other", "t.json") is None
    assert bench.committed_traffic("abc123", "missing.json") is None


def test_committed_records_match_current_sources():
    """The traffic records in profiles/ were taken on the kernel sources as
    they stand (otherwise the benchmark reports no traffic)."""
    for kernel, record in (("decode_pair", "decode_attn_v2_traffic.json"),
                           ("decode_narrow", "decode_narrow_minimind_traffic.json")):
        with open(os.path.join(ROOT, "profiles", record)) as f:
            d = json.load(f)
        assert d["source_hash"] == bench.kernel_source_hash(kernel), record
        assert d["dram_bytes_per_launch"] == d["dram_read_bytes"] + d["dram_write_bytes"]
