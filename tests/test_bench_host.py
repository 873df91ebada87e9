"""Host-side logic of bench.py, without a GPU: the algorithmic byte count of a
launch, the clock summary, the kernel source hash and the lookup of the
committed DRAM traffic figure."""

import os
import shutil

import torch

import bench


def test_strip_c_comments_keeps_code_and_literals():
    src = ('int a = 1; // line comment\n'
           'const char* s = "x // not a comment /* nor this */"; /* block\n   two lines */ int b;\n'
           "char c = '/'; char q = '\\''; const char* e = \"esc \\\" // still a string\"; // gone\n")
    out = bench.strip_c_comments(src)
    assert out == ('int a = 1; \n'
                   'const char* s = "x // not a comment /* nor this */"; \n int b;\n'
                   "char c = '/'; char q = '\\''; const char* e = \"esc \\\" // still a string\"; \n")
    assert bench.strip_c_comments("x /* open to the end") == "x "


def _copy_sources(tmp_path):
    for rel in bench.KERNEL_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), dst)


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    f = tmp_path / bench.KERNEL_SOURCES[0]
    text = f.read_text()
    f.write_text(text + "\n// a remark\n/* and\n   another */\n")
    assert bench.kernel_source_hash() == h0
    f.write_text(text.replace("//", "// edited:", 1))
    assert bench.kernel_source_hash() == h0
    f.write_text(text.replace("kMaxChunks = 16", "kMaxChunks = 17", 1))
    assert bench.kernel_source_hash() != h0


def test_measured_traffic_only_for_the_current_sources(tmp_path, monkeypatch):
    tf = tmp_path / "traffic.txt"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tf))
    assert bench.measured_traffic(4096) is None  # no file
    tf.write_text(f"# comment: ignored\nkernel_source_hash: {bench.kernel_source_hash()}\n"
                  "dram_bytes_per_launch: 1000\nrows_per_launch: 8\n")
    assert bench.measured_traffic(8) == 1000.0
    assert bench.measured_traffic(32) == 4000.0  # scaled by the rows of the launch
    tf.write_text("kernel_source_hash: 0000000000000000\ndram_bytes_per_launch: 1000\nrows_per_launch: 8\n")
    assert bench.measured_traffic(8) is None  # counters of other sources


def test_committed_traffic_matches_the_committed_kernel():
    # the committed ncu figure belongs to the committed sources
    assert bench.measured_traffic(4096) is not None


def test_algorithmic_bytes_counts_valid_and_padding_rows():
    V, K = 1000, 4
    resp = torch.tensor([0, -1, 1, 0], dtype=torch.int32)
    b = dict(V=V, K=K, row_response=resp, rec_count=None)
    assert bench.algorithmic_bytes(b) == 3 * (4 * V + 84) + 8 * 3 * K + 1 * (2 * V + 76)
    # ragged counts: valid rows only, each clamped to [0, K], plus the count itself
    b["rec_count"] = torch.tensor([2, 7, 9, -1], dtype=torch.int32)
    assert bench.algorithmic_bytes(b) == 3 * (4 * V + 84) + 8 * (2 + 4 + 0) + 4 * 3 + 1 * (2 * V + 76)


def test_clock_summary_median_max_and_reasons():
    cs = bench.ClockSampler(0)
    cs.lines = ["1980, 2070, 900.1, Not Active, Not Active, Not Active, Not Active",
                "2070, 2070, 1350.0, Not Active, Not Active, Not Active, Active",
                "2055, 2070, 1300.0, Not Active, Not Active, Not Active, Not Active",
                "[N/A], 2070, 0, Not Active, Not Active, Not Active, Not Active",
                "garbage"]
    s = cs.summary()
    assert s == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    cs.lines = ["2070, 2070, 900, Active, Not Active, Active, Not Active"]
    assert cs.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    cs.lines = []
    assert cs.summary()["reasons"] == ["no samples"]
