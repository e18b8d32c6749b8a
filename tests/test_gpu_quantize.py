"""GPU parity of the Stage-3 quantiser (lynx_quantize_magnitudes, the same
device code the encoder uses) against the oracle's float64 compander, on
values chosen at and around every rounding edge -- including the band where the
kernel switches from its log2 estimate to the exact threshold decision -- and
on a dense uniform sample.  Codes must match except where the oracle's Y lies
within 1e-5 of an edge."""
import numpy as np
import pytest
import torch

from oracle import lynx_oracle as lo
from progressive_kv_quantization_gb300 import lynx as L

pytestmark = pytest.mark.gpu

ALPHAS = [0.25, 1.0, 100.0, 255.0, 1e4, 1e6]


def edge_values(alpha):
    a32 = np.float32(alpha)
    vals = []
    for k in range(1, 128):
        e = np.float32(lo.expander(k - 0.5, float(a32)))
        # float32 neighbours of the edge, from 1 to 3000 ulps away
        for m in (0, 1, 2, 3, 5, 10, 30, 100, 300, 1000, 3000):
            vals.append(np.nextafter(e, np.float32(np.inf), dtype=np.float32) if m == 0 else
                        np.float32(e + m * np.spacing(e)))
            vals.append(np.float32(e - m * np.spacing(e)))
        # points whose Y sits 1e-5 .. 4e-3 from the edge (inside and outside the exact band)
        for dy in (1e-5, 3e-5, 1e-4, 2e-4, 5e-4, 1e-3, 2e-3, 4e-3):
            for sgn in (-1, 1):
                vals.append(np.float32(lo.expander(k - 0.5 + sgn * dy, float(a32))))
    return np.clip(np.array(vals, dtype=np.float32), 0, 1)


@pytest.mark.parametrize("alpha", ALPHAS)
def test_codes_at_and_around_every_edge(cuda_device, alpha):
    rng = np.random.default_rng(int(alpha * 7) % 1000)
    a = np.concatenate([edge_values(alpha), rng.random(1 << 20, dtype=np.float32),
                        np.array([0.0, 1.0, 1e-30, 1e-8, np.float32(1) - np.float32(2 ** -24)], dtype=np.float32)])
    got = L.lynx_quantize_magnitudes(torch.from_numpy(a).cuda(), L.Params(alpha=alpha)).cpu().numpy().astype(np.int64)
    Y, I, _ = lo.quantise(a, np.float32(alpha))
    diff = got != I
    near = np.abs(Y - np.floor(Y) - 0.5) < 1e-5
    assert not np.any(diff & ~near), f"{int((diff & ~near).sum())} codes differ away from an edge"
    assert np.all(np.abs(got - I) <= 1)
    assert got.min() >= 0 and got.max() <= 127


def test_ragged_lengths(cuda_device):
    for n in (1, 7, 9, 1000, 12345):
        a = np.linspace(0, 1, n, dtype=np.float32)
        got = L.lynx_quantize_magnitudes(torch.from_numpy(a).cuda()).cpu().numpy()
        Y, I, _ = lo.quantise(a, np.float32(100.0))
        near = np.abs(Y - np.floor(Y) - 0.5) < 1e-5
        assert np.all((got == I) | near)
