"""bench.py's roofline arithmetic, checked on the host.

Algorithmic bytes are the cache read once (sum_b L_b rows of d_c + d_R bf16
values); algorithmic FLOPs are the two contractions per token and head,
2 n_h (d_c + d_R) for the score and 2 n_h d_c for the weighted sum.  The
DeepSeek-V3 batch (16 x 4096 tokens, 128 heads, 576-wide rows) must give
75 497 472 B and 18 253 611 008 FLOP, i.e. 9.44 us at 8 TB/s and 8.11 us
at 2.25 PFLOP/s.
"""
import json
import os
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _wl(seqlens, n_heads=128, d_latent=512, d_rope=64):
    return SimpleNamespace(seqlens=seqlens, n_heads=n_heads, d_latent=d_latent, d_rope=d_rope)


def test_v3_batch_bytes_and_flops():
    a = bench.algorithmic(_wl([4096] * 16))
    assert a["tokens"] == 65536
    assert a["bytes"] == 65536 * 576 * 2 == 75_497_472
    assert a["flops"] == 65536 * 2 * 128 * (576 + 512) == 18_253_611_008
    assert round(a["bytes"] / 8e12 * 1e6, 2) == 9.44
    assert round(a["flops"] / 2.25e15 * 1e6, 2) == 8.11


def test_ragged_and_low_head_batches():
    a = bench.algorithmic(_wl([1, 0, 129, 4096]))
    assert a["bytes"] == (1 + 129 + 4096) * 1152
    b = bench.algorithmic(_wl([100, 200], n_heads=16))
    assert b["flops"] == 300 * 2 * 16 * 1088 and b["bytes"] == 300 * 1152


def test_peaks_fall_back_only_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6400.0 and p["bf16_tflops"] == 1800.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6490.8, "bf16_tflops": 2100.0}))
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["hbm_gbs"] == 6490.8 and p["bf16_tflops_sustained"] == 2100.0


def test_traffic_is_reported_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    rec = {"source_hash": "abc", "dram_bytes_per_launch": 97.86e6}
    (tmp_path / "profiles" / "decode_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "decode_source_hash", lambda: "abc")
    assert bench.measured_traffic() == pytest.approx(97.86e6)
    monkeypatch.setattr(bench, "decode_source_hash", lambda: "changed")
    assert bench.measured_traffic() is None


def test_traffic_record_is_computed_from_the_ncu_export(tmp_path, monkeypatch):
    raw = "\n".join([
        '"ID","Kernel Name","Block Size","dram__bytes_read.sum","dram__bytes_write.sum"',
        '"","","","Mbyte","Kbyte"',
        '"0","mla::(anonymous namespace)::decode_tc_kernel(CUtensorMap, CUtensorMap)","(384, 1, 1)","605.24","3,579.39"',
        '"1","void mla::(anonymous namespace)::combine_tc_kernel<false>(mla::DecodeLaunch)","(128, 1, 1)","19.01","0"',
    ])
    per = bench.traffic_from_ncu_raw(raw)
    assert per["decode_tc_kernel"]["read"] == pytest.approx(605.24e6)
    assert per["decode_tc_kernel"]["write"] == pytest.approx(3579.39e3)
    assert per["combine_tc_kernel"]["read"] == pytest.approx(19.01e6) and per["combine_tc_kernel"]["write"] == 0
    (tmp_path / "profiles").mkdir()
    (tmp_path / "raw.csv").write_text(raw)
    (tmp_path / "hash.txt").write_text("0123456789abcdef\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = bench.write_traffic_record(str(tmp_path / "raw.csv"), str(tmp_path / "hash.txt"), "ncu ...")
    assert rec["source_hash"] == "0123456789abcdef"
    assert rec["dram_bytes_per_launch"] == pytest.approx(605.24e6 + 3579.39e3 + 19.01e6)
    monkeypatch.setattr(bench, "decode_source_hash", lambda: "0123456789abcdef")
    assert bench.measured_traffic() == pytest.approx(rec["dram_bytes_per_launch"])
