"""The roofline `traffic` that bench.py reports for the gate/up GEMV comes from
a committed ncu summary (profiles/gate_up_gemv_traffic.txt) and holds only
while the kernel sources hash to the value recorded beside it.  These checks
keep that figure honest: the summary is current for the sources in the tree,
its DRAM bytes are within a fraction of a percent of the kernel's algorithmic
bytes (no weight byte read twice), and a summary for other sources is refused."""

import os

import bench

ALGORITHMIC = 2 * (18944 * 3584 // 2 + 18944 * 3584 // 64) + 6 * 3584 + 2 * 18944   # 70,076,416 bytes


def test_recorded_traffic_is_for_the_sources_in_the_tree():
    t = bench.recorded_traffic()
    assert t is not None, "the gate/up traffic summary was taken on other kernel sources: re-capture it"
    assert ALGORITHMIC == 70076416
    assert ALGORITHMIC <= t <= 1.01 * ALGORITHMIC


def test_a_summary_for_other_sources_is_refused(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "profiles", "gate_up_gemv_traffic.txt")
    text = open(src).read().replace("source_hash = " + bench.kernel_source_hash(), "source_hash = 0000000000000000")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "gate_up_gemv_traffic.txt").write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "e" * 16)
    assert bench.recorded_traffic() is None
