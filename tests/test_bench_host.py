"""Host-side pieces of bench.py that need no GPU: reading the measured peak,
and the algorithmic byte counts of a decode launch."""
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
