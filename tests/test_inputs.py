"""The seeded input generators: BF16 rounding, shapes, outlier sets, determinism."""
import json
import os

import numpy as np
import torch

from progressive_kv_quantization_gb300 import inputs


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 37
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 65504.0]      # ties, signed zero
    ours = inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(inputs.bf16_bits_to_f32(ours), torch.from_numpy(ours.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_pages_shape_outliers_and_determinism():
    m = inputs.outlier_pairs(8, 0)
    assert m.shape == (8, 128) and m.sum() == 10            # 1% of 1024 pairs
    assert inputs.outlier_pairs(4, 0).sum() == 5
    assert inputs.outlier_pairs(1, 0, count=4).sum() == 4
    p = inputs.kv_pages_np(2, 512, 7, inputs.outlier_pairs(2, 7))
    assert p.shape == (4, 128, 256) and p.dtype == np.uint16
    assert np.array_equal(p, inputs.kv_pages_np(2, 512, 7, inputs.outlier_pairs(2, 7)))
    x = inputs.bf16_bits_to_f32(p)
    # outlier channels are ~100x larger than the rest
    mask = inputs.outlier_pairs(2, 7)
    rows = x.reshape(2, 2, 128, 256)
    big = np.abs(rows[mask[:, None, :].repeat(2, 1)]).mean()
    small = np.abs(rows[~mask[:, None, :].repeat(2, 1)]).mean()
    assert big > 30 * small


def test_normalised_values_concentrate_as_in_figure_5():
    """Figure 5 of the paper: about half of the normalised values lie in the
    middle 17% of [-1, 1].  The synthetic data should look alike (loose check)."""
    from oracle import lynx_oracle as lo
    with open(os.path.join(os.path.dirname(__file__), "golden", "printed_values.json")) as f:
        g = json.load(f)["figure5_concentration"]
    p = inputs.kv_pages_np(8, 1024, 1, inputs.outlier_pairs(8, 1))
    st = lo.run_stages(p, 100.0, np.float32(1e-6))
    frac = float(np.mean(np.abs(st.xfinal) <= g["half_width"]))
    assert 0.3 < frac < 0.7
