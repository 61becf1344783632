"""Host-side check of bench.py's bookkeeping (no GPU): the kernel-source hash
that ties the committed ncu traffic figure to the kernels it was taken on
ignores comments but not code."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    src = os.path.join(ROOT, "int4_weight_only_g128_gb300", "csrc", "w4g128_ptx.cuh")
    copy = tmp_path / "k.cuh"
    shutil.copy(src, copy)
    monkeypatch.setattr(bench, "KERNEL_SOURCES", [str(copy)])
    base = bench.kernel_source_sha()
    text = copy.read_text()
    copy.write_text("// a new comment line\n\n" + text.replace("\n", "  // trailing remark\n", 1))
    assert bench.kernel_source_sha() == base
    copy.write_text(text.replace("return t;", "return t + 0ull;", 1))
    assert bench.kernel_source_sha() != base

