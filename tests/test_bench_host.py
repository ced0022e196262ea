"""Host logic of bench.py that decides whether `roofline.traffic` may be reported (CPU only).

`traffic` comes from a committed ncu summary only while the summary's recorded source hash
matches the current kernel sources. The hash must ignore comments (editing a comment does
not change the generated code) and must change with any code edit; the lookup must return
the stamped bytes for a matching hash and nothing otherwise.
"""
import os
import shutil

import bench

SRC = os.path.join(bench.ROOT, "fp4_communication_compression_gb300", "csrc")
HDR = os.path.join(bench.ROOT, "include", "fp4q.h")


def _tree(tmp_path):
    csrc = tmp_path / "fp4_communication_compression_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in os.listdir(SRC):
        if f.endswith((".cu", ".cuh")):
            shutil.copy(os.path.join(SRC, f), csrc / f)
    (tmp_path / "include").mkdir()
    shutil.copy(HDR, tmp_path / "include" / "fp4q.h")
    return csrc / "fp4q.cu"


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    cu = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_sha()
    assert h0 == bench.kernel_source_sha()
    text = cu.read_text()
    cu.write_text("// a new line comment\n" + text + "\n/* a block\n   comment */\n\n")
    assert bench.kernel_source_sha() == h0
    cu.write_text(text + "\nstatic int g_unused_probe;\n")
    assert bench.kernel_source_sha() != h0


def test_ncu_traffic_needs_a_matching_stamp(tmp_path, monkeypatch):
    _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("compress_kernel") is None          # no profiles/ at all
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = bench.kernel_source_sha()
    (prof / "compress_x.md").write_text(
        f"text\nbench-traffic kernel=compress_kernel source_sha256={sha} dram_bytes_per_launch=12345\n")
    (prof / "reduce_x.md").write_text(
        "bench-traffic kernel=reduce_kernel source_sha256=0123456789abcdef dram_bytes_per_launch=999\n")
    assert bench.ncu_traffic("compress_kernel") == 12345
    assert bench.ncu_traffic("reduce_kernel") is None              # taken on other sources
    assert bench.ncu_traffic("decompress_kernel") is None          # no summary


def test_committed_summaries_carry_stamps():
    """Every per-kernel summary of the bench workload records its kernel and source hash."""
    names = [n for n in os.listdir(os.path.join(bench.ROOT, "profiles"))
             if n.endswith("_tp_activation_4096x4096.md")]
    assert names
    for n in names:
        text = open(os.path.join(bench.ROOT, "profiles", n)).read()
        assert "bench-traffic kernel=" in text and "source_sha256=" in text, n
