"""Host-side helpers of bench.py (no GPU): the attention FLOP count and the
roofline denominators."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_attention_flops_closed_form():
    import bench
    # Q K^T and P V: 2 * 128 multiply-adds each per query row and key
    assert bench.attn_flops(1, 1, 1, 1, 1) == pytest.approx(4 * 128)
    B, T, G, Hkv, keys = 64, 8, 4, 8, 16384
    assert bench.attn_flops(B, T, G, Hkv, keys) == pytest.approx(4.0 * 128 * T * G * keys * Hkv * B)


def test_peaks_read_the_measured_file_or_fall_back(tmp_path, monkeypatch):
    import bench
    p = tmp_path / "MEASURED_PEAKS.json"
    p.write_text(json.dumps({"hbm_gbs": 1234.5, "bf16_tflops": 999.0}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (1234.5, "measured")
    assert bench.tensor_peak() == (999.0, "measured")
    p.unlink()
    assert bench.peaks()[1] == "fallback" and bench.tensor_peak()[1] == "fallback"
    assert bench.NOMINAL_HBM_GBS == 8000.0
