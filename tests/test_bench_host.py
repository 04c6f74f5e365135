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


def test_traffic_scales_a_small_capture_of_the_current_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("state_7b", 7_000_000_000) == (None, None)
    d = bench.kernel_source_digest()
    (prof / "dram_state_7b.txt").write_text(
        f"kernel_source_digest: {d}\nzero1_adamw_ag_kernel.dram_bytes_per_param: 32.5\n")
    assert bench.kernel_traffic("state_7b", 1000) == (32500.0, "profiles/dram_state_7b.txt")
    assert bench.kernel_traffic("state_7b@5000", 5000)[0] == 162500.0     # a resized recipe uses its own summary
    (prof / "dram_state_7b.txt").write_text("kernel_source_digest: 0\nzero1_adamw_ag_kernel.dram_bytes_per_param: 1\n")
    assert bench.kernel_traffic("state_7b", 1000) == (None, None)          # taken on other sources: not used


def test_measured_peak(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 1234.5}))
    assert bench.measured_peak() == (1234.5, "measured")


def test_digest_covers_the_kernel_sources_only():
    """The digest that ties ncu summaries to the code covers what the kernels
    compile from, and not host-side launch policy (zero1_policy.h), whose
    retuning changes no kernel."""
    names = sorted(os.path.basename(p) for p in bench.KERNEL_SRCS)
    assert names == ["zero1_internal.h", "zero1_kernels.cu", "zero1_ptx.cuh"]
    kernels = open(os.path.join(bench.CSRC, "zero1_kernels.cu")).read()
    assert '#include "zero1_policy.h"' not in kernels
