"""bench.py's host logic on CPU: the kernel-source digest that ties committed
ncu summaries to the code, the traffic lookup, and the measured-peak read."""
from __future__ import annotations

import json
import os
import shutil

import bench


def test_digest_ignores_comments_and_whitespace(tmp_path):
    src = os.path.join(bench.CSRC, "zero1_kernels.cu")
    a = tmp_path / "a.cu"
    shutil.copy(src, a)
    base = bench.kernel_source_digest([str(a)])
    text = a.read_text()
    a.write_text("// a new comment\n" + text.replace("\n", "\n  \n", 3) + "\n/* trailing\n block */\n")
    assert bench.kernel_source_digest([str(a)]) == base
    a.write_text(text.replace("kVec", "kVec ", 1).replace("constexpr int kStages = 4;", "constexpr int kStages = 5;"))
    assert bench.kernel_source_digest([str(a)]) != base


def test_traffic_comes_only_from_summaries_of_the_current_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("gpt2_small") == (None, None)
    d = bench.kernel_source_digest()
    (prof / "zero1_adamw_ag_kernel_gpt2_small.txt").write_text(
        f"kernel_source_digest: {d}\ndram_bytes_per_launch: 123\n")
    assert bench.kernel_traffic("gpt2_small") == (123.0, "profiles/zero1_adamw_ag_kernel_gpt2_small.txt")
    (prof / "dram_gpt2_small.txt").write_text(
        f"kernel_source_digest: {d}\nzero1_adamw_ag_kernel.dram_bytes_per_launch: 456\n")
    assert bench.kernel_traffic("gpt2_small") == (456.0, "profiles/dram_gpt2_small.txt")    # full size first
    (prof / "dram_gpt2_small.txt").write_text("kernel_source_digest: 0\nzero1_adamw_ag_kernel.dram_bytes_per_launch: 1\n")
    assert bench.kernel_traffic("gpt2_small")[0] == 123.0                                  # stale one skipped


def test_measured_peak(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 1234.5}))
    assert bench.measured_peak() == (1234.5, "measured")
