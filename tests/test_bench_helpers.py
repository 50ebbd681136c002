"""CPU checks of the benchmark's roofline arithmetic and of how it reads the
committed ncu summaries (no GPU involved)."""

import hashlib
import os

import pytest

import bench


def test_hbm_roofline_arithmetic():
    peaks = {"hbm_gbs": 6000.0}
    r = bench.hbm_roofline("k", alg_bytes=3_000_000_000, out_bytes=600_000_000, kernel_ms=0.5,
                           peaks=peaks, peak_kind="measured", traffic=3.1e9)
    # 3 GB in 0.5 ms = 6000 GB/s = the whole peak; the output bytes are reported beside it
    assert r["achieved"] == pytest.approx(6000.0)
    assert r["frac"] == pytest.approx(1.0)
    assert r["frac_incl_output"] == pytest.approx(1.2)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["traffic"] == 3.1e9
    assert r["algorithmic_bytes_per_launch"] == 3_000_000_000 and r["kernel_ms"] == 0.5


def test_l2_stream_arithmetic(monkeypatch):
    # the L2 side of the sparse prefill line: bytes out of L2 per launch over the
    # kernel time, against the rate the diagnostic measured in the same run
    monkeypatch.setattr(bench, "measure_l2_read", lambda: {"gbs": 20000.0, "how": "stub"})
    r = bench.l2_stream(4_000_000_000, 0.5, "k records")
    assert r["achieved_gbs"] == pytest.approx(8000.0)
    assert r["peak_gbs"] == 20000.0 and r["frac"] == pytest.approx(0.4)
    assert r["bytes_per_launch"] == 4_000_000_000 and r["bytes"] == "k records" and r["peak_source"] == "stub"


def test_profiled_traffic_only_for_the_profiled_source(tmp_path, monkeypatch):
    src = tmp_path / "sparse_attention_indexer_fp8_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text("kernel v1\n")
    h = hashlib.sha256(b"kernel v1\n").hexdigest()[:16]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "p.md").write_text(f"# p\n\n- source_sha256_16: `{h}`\n- dram_bytes_per_launch: `123456`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "PROFILE_DIR", str(prof))
    assert bench.profiled_traffic("p.md", "k.cu") == 123456.0
    (src / "k.cu").write_text("kernel v2\n")          # the kernel changed since the capture
    assert bench.profiled_traffic("p.md", "k.cu") is None
    assert bench.profiled_traffic("missing.md", "k.cu") is None


def test_committed_profiles_match_the_sources():
    # every summary that carries a source hash and a traffic figure was taken on
    # the kernel source as committed, so the bench lines report that traffic
    names = [n for n in os.listdir(bench.PROFILE_DIR) if n.endswith(".md")]
    with_traffic = []
    for n in names:
        text = open(os.path.join(bench.PROFILE_DIR, n)).read()
        if "- dram_bytes_per_launch:" in text and "logits" in text.split("\n")[0]:
            with_traffic.append(n)
    assert with_traffic, "no scoring-kernel profile with a traffic figure"
    for n in with_traffic:
        assert bench.profiled_traffic(n, "logits.cu") is not None, n
