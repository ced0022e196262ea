"""Host logic of bench.py that decides whether `roofline.traffic` may be reported (CPU only).

`traffic` comes from a committed ncu summary only while the summary's recorded source hash
matches the current kernel sources. The hash must ignore comments (editing a comment does
not change the generated code) and must change with any code edit; the lookup must return
the stamped bytes for a matching hash and nothing otherwise.
"""
import os
import re
import shutil

import pytest

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
    """Every committed summary that feeds `roofline.traffic` records its kernel, source hash
    and bytes in the stamp format the bench reads."""
    pdir = os.path.join(bench.ROOT, "profiles")
    stamped = [n for n in os.listdir(pdir) if n.endswith(".md") and "bench-traffic" in open(os.path.join(pdir, n)).read()]
    assert stamped
    for n in stamped:
        text = open(os.path.join(pdir, n)).read()
        assert re.search(r"bench-traffic kernel=\w+ source_sha256=[0-9a-f]{16} dram_bytes_per_launch=\d+", text), n


def test_both_arms_print_the_same_config(monkeypatch, capsys):
    """The reference arm's config dict is the GPU arm's (bench_config), so the two lines
    describe one workload; its sample is bounded."""
    import json

    import numpy as np
    small = np.arange(4096, dtype=np.uint16) % 200 + 0x3c00
    monkeypatch.setattr(bench, "headline_inputs", lambda: (small, small[::-1].copy()))
    monkeypatch.setattr(bench, "REF_SAMPLE", 2048)

    class A:
        steps, warmup = 2, 1
    assert bench.reference_arm(A(), rank=0, world=1) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.bench_config(1)
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert "l2" not in line["config"]


def test_bench_refuses_to_report_after_a_fault():
    """A set fault word (read from a stand-in of the binding) stops the report."""
    import pytest

    class FakeFq:
        def __init__(self, word):
            self.word, self.cleared = word, False

        def fault_flags(self, clear=False):
            w = self.word
            if clear:
                self.word, self.cleared = 0, True
            return w

    ok = FakeFq(0)
    bench.require_no_fault(ok, "steps")
    assert ok.cleared
    with pytest.raises(bench.FaultWordSet, match="0x1"):
        bench.require_no_fault(FakeFq(1), "steps")
    with pytest.raises(bench.FaultWordSet, match="0x6"):
        bench.require_no_fault(FakeFq(6), "steps")


def test_alg_bytes_table():
    assert bench.alg_bytes("compress") == 2.578125
    assert bench.alg_bytes("decompress_bf16_b1") == 4.578125
    assert bench.alg_bytes("roundtrip") == 4.0
    assert bench.alg_bytes("reduce_r4") == 5 * 0.578125
    assert bench.alg_bytes("compress", group=32) == 2 + 0.5 + 1 / 32 + 4 / 256
    assert bench.alg_bytes("compress", scales="e8m0") == 2.53125


def test_ncu_traffic_scales_a_smaller_capture(tmp_path, monkeypatch):
    _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = bench.kernel_source_sha()
    (prof / "d.md").write_text(
        f"bench-traffic kernel=decompress_kernel source_sha256={sha} dram_bytes_per_launch=1000 elements=256\n")
    assert bench.ncu_traffic("decompress_kernel", 1024) == 4000
    assert bench.ncu_traffic("decompress_kernel") == 1000


def test_target_summary_counts_only_large_workloads():
    cfg = {"small": {"bytes_bf16": 1 << 20, "kernels": [{"kernel": "compress", "frac_of_peak": 0.1}]},
           "big": {"bytes_bf16": 1 << 27, "kernels": [{"kernel": "compress", "frac_of_peak": 0.75},
                                                      {"kernel": "roundtrip", "frac_of_peak": 0.65,
                                                       "group": 32, "fwht": 0}]}}
    s = bench.target_summary(cfg)
    assert s["records"] == 2 and s["met"] == 1
    assert s["below"] == [{"big:roundtrip_g32_fwht0": 0.65}]
    assert "back_to_back" not in s          # no record carries a back-to-back time


def test_target_summary_counts_back_to_back_times_apart():
    cfg = {"big": {"bytes_bf16": 1 << 26, "kernels": [
        {"kernel": "compress", "frac_of_peak": 0.68, "stream_frac_of_peak": 0.74},
        {"kernel": "reduce_r4", "frac_of_peak": 0.5, "stream_frac_of_peak": 0.59},
        {"kernel": "compress", "frac_of_peak": 0.74, "stream_frac_of_peak": 0.74,
         "variant": "compress_tc (fwht=2, relaxed parity)"}]}}
    s = bench.target_summary(cfg)
    assert s["records"] == 2 and s["met"] == 0
    assert s["back_to_back"] == {"records": 2, "met": 1, "below": [{"big:reduce_r4": 0.59}], "min_frac": 0.59}


def test_back_to_back_buffer_sets_cover_three_times_l2():
    class Props:
        L2_cache_size = 100

    class FakeCuda:
        @staticmethod
        def get_device_properties(dev):
            return Props()

    class FakeTorch:
        cuda = FakeCuda

    t = bench.Timer.__new__(bench.Timer)
    t.torch, t.dev = FakeTorch, None
    assert t.buffer_sets(100) == 3 and t.buffer_sets(101) == 3 and t.buffer_sets(99) == 4
    assert t.buffer_sets(1000) == 2          # never fewer than two sets
    rec = bench.kernel_record("compress", 1 << 20, 1.0, 1000.0, stream_ms=0.5)
    assert rec["stream_us"] == 500.0 and rec["stream_frac_of_peak"] == 2 * rec["frac_of_peak"]


def test_back_to_back_hold_doubles_until_the_host_keeps_up():
    """The start event must still be pending when the host has enqueued the region's last
    launch; a region where it was not is taken again with twice the hold."""
    log = []

    class Event:
        n = 0

        def __init__(self, enable_timing=True):
            pass

        def record(self, stream):
            pass

        def query(self):              # passed already while the hold is below 2^24 cycles
            return state["hold"] < (1 << 24)

        def elapsed_time(self, other):
            return 8.0

    state = {"hold": 0}

    class FakeCuda:
        @staticmethod
        def _sleep(cycles):
            state["hold"] = cycles
            log.append(cycles)

        @staticmethod
        def synchronize(dev=None):
            pass

    FakeCuda.Event = Event

    class FakeTorch:
        cuda = FakeCuda

    t = bench.Timer.__new__(bench.Timer)
    t.torch, t.dev, t.stream = FakeTorch, None, None
    t.hold_cycles = 1 << 22
    t.flush = lambda: None
    calls = []
    ms = t.stream_ms([lambda: calls.append(0)] * 2, reps=3, rounds=2)
    assert ms == 2.0                              # 8 ms over 2 rounds x 2 launches
    assert log == [1 << 22, 1 << 23, 1 << 24, 1 << 24, 1 << 24]
    assert t.hold_cycles == 1 << 24
    # a host that never keeps up ends in an error, not in a starved number
    Event.query = lambda self: True
    t.hold_cycles = 1 << 29
    with pytest.raises(RuntimeError, match="longest hold"):
        t.stream_ms([lambda: None], reps=1, rounds=1)


def test_target_summary_lists_the_e8m0_variant_apart():
    cfg = {"F2": {"bytes_bf16": 1 << 27, "kernels": [
        {"kernel": "compress", "frac_of_peak": 0.6, "stream_frac_of_peak": 0.7,
         "variant": "e8m0 (microscaled scales)"}]},
           "C5": {"bytes_bf16": 1 << 27, "kernels": [{"kernel": "compress", "frac_of_peak": 0.8}]}}
    s = bench.target_summary(cfg)
    assert s["records"] == 1 and s["met"] == 1
    assert s["e8m0_variant"] == [{"F2:compress": [0.6, 0.7]}]
    rec = bench.kernel_record("compress", 1 << 20, 1.0, 1000.0, 32, "e8m0")
    assert rec["alg_bytes_per_elem"] == 2.53125
