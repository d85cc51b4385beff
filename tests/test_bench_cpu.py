"""Host-side helpers of the benchmark (no GPU): the kernel list of a call,
the peak figures it divides by, and the ncu traffic figure it reports only
for the kernel source the capture was taken on."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_mla_speculative_gb300 import binding as mb  # noqa: E402


def test_kernel_list_follows_the_pack_schedule():
    assert bench.kernels_of(mb.KERNEL_TC, 2, "idle_sms") == \
        "pack_kv_overlap_kernel + partial_tc_kernel + combine_kernel"
    assert bench.kernels_of(mb.KERNEL_TC, 2, "whole") == "pack_kv_kernel + partial_tc_kernel + combine_kernel"
    assert bench.kernels_of(mb.KERNEL_TC, 1, "whole") == "pack_kv_kernel + partial_tc_kernel"
    assert bench.kernels_of(mb.KERNEL_TC, 3, "none") == "partial_tc_kernel + combine_kernel"
    assert bench.kernels_of(mb.KERNEL_MMA, 3) == "partial_mma_kernel + combine_kernel"
    assert bench.kernels_of(mb.KERNEL_PAIR, 19, "whole") == \
        "pack_kv_kernel + partial_pair_kernel + combine_kernel"
    assert bench.kernels_of(mb.KERNEL_PAIR, 2, "idle_sms") == \
        "pack_kv_overlap_kernel + partial_pair_kernel + combine_kernel"


def test_peaks_fall_back_without_a_measurement(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6000.0, "bf16_tflops": 1800.0}))
    peaks, src = bench.load_peaks()
    assert src == "measured" and peaks["hbm_gbs"] == 6000.0 and peaks["bf16_tflops"] == 1800.0


def test_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    src_hash = bench.kernel_source_hash("partial_pair_kernel")
    assert src_hash != bench.kernel_source_hash("partial_tc_kernel")
    prof = tmp_path / "profiles"
    prof.mkdir()
    entry = {"workload": "decode_batch", "dram_bytes_per_launch": 123.0, "source_sha1": src_hash}
    (prof / "traffic.json").write_text(json.dumps({"partial_pair_kernel": entry}))
    # the hash is taken from the real sources; only the traffic file is redirected
    real_root = bench.ROOT
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel="partial_pair_kernel": src_hash)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("decode_batch", "partial_pair_kernel") == 123.0
    assert bench.profiled_traffic("decode_batch", "partial_tc_kernel") is None
    assert bench.profiled_traffic("tree", "partial_pair_kernel") is None
    entry["source_sha1"] = "0" * 40
    (prof / "traffic.json").write_text(json.dumps({"partial_pair_kernel": entry}))
    assert bench.profiled_traffic("decode_batch", "partial_pair_kernel") is None
    monkeypatch.setattr(bench, "ROOT", real_root)
