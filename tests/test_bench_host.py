"""Host-side pieces of bench.py that need no GPU: reading the measured peak,
the algorithmic byte and flop counts of the decode and multi-token launches,
the DRAM-traffic record that is valid only for the kernel source it was
taken on, and the clock summary of the timed window."""
import json

import numpy as np
import pytest

import bench


@pytest.mark.parametrize("content,want", [
    ('{"hbm_gbs": 6781.2}', (6781.2, "measured")),
    ('{"hbm_gbs": {"value": 6700}}', (6700.0, "measured")),
    ('{"gb300": {"hbm_gbs": 6600, "bf16_tflops": 1900}}', (6600.0, "measured")),
    ('[1, 2]', (bench.FALLBACK_HBM_GBS, "fallback")),
    ('{"hbm_gbs": "n/a"}', (bench.FALLBACK_HBM_GBS, "fallback")),
    ('not json', (bench.FALLBACK_HBM_GBS, "fallback")),
])
def test_measured_peak_file_shapes(tmp_path, monkeypatch, content, want):
    (tmp_path / "MEASURED_PEAKS.json").write_text(content)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.hbm_peak() == want


def test_missing_peak_file_falls_back(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.hbm_peak() == (bench.FALLBACK_HBM_GBS, "fallback")


def test_decode_bytes_formula():
    """K + V of every context token once, Q and out, table entries read and lengths."""
    lens = np.array([1, 16, 17, 100])
    Hq, Hkv, D = 8, 2, 128
    kv = int(lens.sum()) * Hkv * D * 2 * 2
    tables = int(((lens + 15) // 16).sum()) * 4 + len(lens) * 4
    io = len(lens) * Hq * D * (2 + 4)
    assert bench.decode_bytes(lens, Hq, Hkv, D, 2, 2, 4) == kv + tables + io
    # 1-byte codes add two float32 scales per token
    assert bench.decode_bytes(lens, Hq, Hkv, D, 1, 2, 4) == kv // 2 + int(lens.sum()) * 8 + tables + io


class _PrefillShape:
    def __init__(self, lens, qlens, Hq=4, Hkv=2, D=64, kv_dtype="f16"):
        self.context_lens, self.q_lens = lens, qlens
        self.Hq, self.Hkv, self.D, self.kv_dtype = Hq, Hkv, D, kv_dtype
        self.T = int(sum(qlens))


@pytest.mark.parametrize("kv", ["f16", "fp8"])
def test_prefill_cost_by_brute_force(kv):
    """Bytes: K+V of every context token once (+ two float32 scales per token for
    1-byte caches), 16-bit q and out rows, table entries, lengths and q_start;
    flops: 4 * D per (query row, visible key), counted key by key."""
    lens, qlens = [1, 16, 17, 40, 5], [1, 3, 17, 40, 0]
    w = _PrefillShape(lens, qlens, kv_dtype=kv)
    e = 1 if kv == "fp8" else 2
    keys = 0
    for L, n in zip(lens, qlens):
        for i in range(n):
            keys += sum(1 for t in range(L) if t <= L - n + i)
    kv_bytes = sum(lens) * w.Hkv * w.D * 2 * e + (sum(lens) * 8 if e == 1 else 0)
    io = w.T * w.Hq * w.D * 2 * 2
    meta = sum((L + 15) // 16 for L in lens) * 4 + len(lens) * 4 + (len(lens) + 1) * 4
    assert bench.prefill_cost(w) == (kv_bytes + io + meta, 4 * w.D * w.Hq * keys)


def test_traffic_record_follows_the_kernel_source(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic_decode_demo.txt").write_text(
        "kernel: x\napi: pa_decode_append\ndram_bytes_per_launch: 12345\nkernel_source_sha256_16: abc\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    assert bench.profiled_traffic("demo", "pa_decode_append") == 12345.0
    assert bench.profiled_traffic("other", "pa_decode_append") is None  # no record for that workload
    # a record of another entry point (the fixed grid against the item list) does not count
    assert bench.profiled_traffic("demo", "pa_decode_append_segments (one-member groups)") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "changed")
    assert bench.profiled_traffic("demo", "pa_decode_append") is None  # stale after a kernel edit


def test_clock_summary_reads_the_timed_window():
    import time as _t
    base = _t.mktime(_t.strptime("2026/12/02 10:00:00", "%Y/%m/%d %H:%M:%S"))
    s = bench.ClockSampler(0)
    s.lines = [
        "2026/12/02 10:00:00.100, 1200, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:01.100, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:01.300, 2060, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:01.500, 2070, 2070, 940.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:03.000, 1000, 2070, 200.0, 0x0, Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    got = s.summary([(base + 1.0, base + 1.6)])
    assert got["samples"] == 3 and got["window"] == "timed region"
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]  # the hw_slowdown sample lies outside the window
    # several windows: the timed region plus a clock hold that covers the late sample
    got = s.summary([(base + 1.0, base + 1.2), (base + 2.9, base + 3.1)], "timed region + hold")
    assert got["samples"] == 2 and got["window"] == "timed region + hold"
    assert got["reasons"] == ["hw_slowdown", "sw_power_cap"]
    # a window between two samples holds none: reported as such, never the whole run
    got = s.summary([(base + 2.0, base + 2.01)])
    assert got["samples"] == 0 and got["sm_mhz"] is None and "no sample inside" in got["window"]
    s.lines = []
    assert s.summary([(0, 1)])["samples"] == 0
