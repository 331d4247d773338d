"""Host-side logic of bench.py that needs no GPU: the fingerprint that ties the
reported DRAM traffic to the kernel sources the ncu capture ran, and the
lookup of that traffic in the committed summary."""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

SRC = os.path.join(ROOT, "bit_block_quantized_q4_gb300", "csrc")


def _reader(edit=None):
    def read(name):
        text = open(os.path.join(SRC, name)).read()
        return edit(name, text) if edit else text
    return read


def test_fingerprint_ignores_comments_and_whitespace():
    base = bench.kernel_fingerprint(_reader())
    commented = bench.kernel_fingerprint(_reader(
        lambda name, t: "// a new comment\n/* and a block\n   comment */\n" + t.replace(";\n", ";  \n", 3)))
    assert commented == base


def test_fingerprint_changes_with_code_in_any_kernel_source():
    base = bench.kernel_fingerprint(_reader())
    for target in bench.KERNEL_SOURCES:
        changed = bench.kernel_fingerprint(_reader(
            lambda name, t, target=target: t + "\nstatic int probe_value = 1;\n" if name == target else t))
        assert changed != base, target


def test_traffic_is_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    fp = bench.kernel_fingerprint()
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the summary's sources match the tree: the captured launch's traffic is
    # scaled to the pass by algorithmic bytes (a 1-layer capture, 64 layers)
    (prof / "gemv_stream_b1_27b_layer.md").write_text(
        f"- dram_bytes_per_launch: 1000\n- algorithmic_bytes_per_launch: 990\n"
        f"- kernel_fingerprint_16: {fp}\n")
    monkeypatch.setattr(bench, "kernel_fingerprint", lambda read=None: fp)
    assert bench.profiled_traffic(990 * 64) == 1000 * 64
    # another fingerprint: the capture is stale and no figure is reported
    (prof / "gemv_stream_b1_27b_layer.md").write_text(
        "- dram_bytes_per_launch: 1000\n- algorithmic_bytes_per_launch: 990\n"
        "- kernel_fingerprint_16: 0000000000000000\n")
    assert bench.profiled_traffic(990 * 64) is None
