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


def test_pm1_fraction_counts_and_checks_edge_differences(tmp_path):
    """The code comparison the bench reports: identical codes give 0; a +-1
    magnitude step on a code whose Y is near an edge is counted and accepted; a
    step away from an edge is flagged."""
    import numpy as np

    import bench
    from oracle import lynx_oracle as lo
    from progressive_kv_quantization_gb300 import inputs
    kb = inputs.kv_pages_np(1, 512, 3, inputs.outlier_pairs(1, 3, count=2))
    a, r, _, st = lo.encode_pages(kb, 100.0, np.float32(1e-6), return_stages=True)
    stages = {"anchor": a, "residual": r, "Y": st.Y}
    f = tmp_path / "g.npz"
    np.savez(f, anchor=a, residual=r)
    d = bench.pm1_fraction(str(f), stages)
    assert d["fraction"] == 0.0 and d["all_at_rounding_edges"] and d["codes_compared"] == a.size * 2

    def with_code(i_new, flat):
        """planes with element `flat` re-encoded at magnitude i_new (same sign)"""
        qa = lo.unpack_nibbles(a).astype(np.int32).ravel()
        qr = lo.unpack_nibbles(r).astype(np.int32).ravel()
        s = 1 if qa[flat] >= 0 else -1
        v = i_new >> 4
        qa[flat] = v if s > 0 else -v - 1
        qr[flat] = 16 * v + 7 - i_new
        shape = (a.shape[0], a.shape[1], 2 * a.shape[2])
        return lo.pack_nibbles(qa.reshape(shape)), lo.pack_nibbles(qr.reshape(shape))

    Y = st.Y.ravel()
    frac = np.abs(Y - np.floor(Y) - 0.5)
    near, far = int(np.argmin(frac)), int(np.argmax(frac))
    I = st.I.ravel()
    for flat, ok in ((near, frac[near] < 1e-5), (far, False)):
        i_new = int(I[flat]) + (1 if I[flat] < 127 else -1)
        ga, gr = with_code(i_new, flat)
        np.savez(f, anchor=ga, residual=gr)
        d = bench.pm1_fraction(str(f), stages)
        assert d["differing"] == 1 and d["all_at_rounding_edges"] == bool(ok)


def test_write_traffic_scales_a_small_capture(tmp_path, monkeypatch):
    """profiles/traffic.json from an ncu CSV: mean read + write bytes of the
    captured launches times the stated scale, keyed by the kernel's sources."""
    import bench
    csv = tmp_path / "cap.csv"
    rows = ['"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"']
    for i, (rd, wr) in enumerate(((100.0, 10.0), (300.0, 30.0))):
        rows.append(f'"{i}","void lynx::encode_kernel<0>()","dram__bytes_read.sum","Mbyte","{rd}"')
        rows.append(f'"{i}","void lynx::encode_kernel<0>()","dram__bytes_write.sum","Mbyte","{wr}"')
        rows.append(f'"{i}","other_kernel","dram__bytes_read.sum","Mbyte","999"')
    csv.write_text("\n".join(rows) + "\n")
    out = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(out))
    bench.write_traffic(str(csv), ["encode=encode_kernel:2.5"])
    d = json.loads(out.read_text())
    assert d["encode"]["bytes_per_launch"] == int((200e6 + 20e6) * 2.5)
    assert d["encode"]["launches_captured"] == 2
    assert d["encode"]["source_sha"] == bench.source_sha(bench.KERNEL_SOURCES["encode"])
