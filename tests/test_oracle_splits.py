"""Pins of oracle/splits.py: the 4+4 split is the paper's split stream exactly;
the other widths satisfy the definition of the 8-bit code, place every bit
where the layout says, and trade Anchor size for Anchor-only error."""
import numpy as np
import pytest

from oracle import baselines as bl
from oracle import lynx_oracle as lo
from oracle import splits as sp
from progressive_kv_quantization_gb300 import inputs

EPS = 1e-6


def _pages(n, seed):
    return inputs.kv_pages_np(1, 256 * n, seed, inputs.outlier_pairs(1, seed))


def test_four_four_split_is_the_paper_split():
    x = _pages(2, 3)
    a, r, m = sp.encode_pages_split(x, 4, 100.0, EPS)
    a0, r0, m0 = lo.encode_pages(x, 100.0, EPS)
    assert np.array_equal(a, a0) and np.array_equal(r, r0) and np.array_equal(m, m0)
    assert np.array_equal(sp.reconstruct_split(a, None, m, 4, 100.0, EPS), lo.reconstruct(a0, None, m0, 100.0, EPS))
    assert np.array_equal(sp.reconstruct_split(a, r, m, 4, 100.0, EPS), lo.reconstruct(a0, r0, m0, 100.0, EPS))


@pytest.mark.parametrize("A", [2, 3, 5, 6])
def test_split_definition_on_every_code(A):
    """For every 8-bit code: the Anchor is q8 >> R (arithmetic), the Residual
    lies in [-2^(R-1), 2^(R-1) - 1], and Anchor + Residual give I back."""
    R = 8 - A
    I = np.tile(np.arange(128), 2)
    S = np.repeat([1, -1], 128)
    qa, qr = sp.split_codes(I, S, A)
    q8 = np.where(S > 0, I, -I - 1)
    assert np.array_equal(qa, q8 >> R)
    assert qr.min() >= -(1 << (R - 1)) and qr.max() <= (1 << (R - 1)) - 1
    V = np.where(qa < 0, -qa - 1, qa)
    assert np.array_equal((V << R) + (1 << (R - 1)) - 1 - qr, I)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6])
def test_bit_positions_brute_force(bits):
    """Token t's code of a 32-token chunk sits at bits bits*t .. of the chunk's
    little-endian bit string, chunks in order; unpack inverts pack."""
    rng = np.random.default_rng(bits)
    codes = rng.integers(-(1 << (bits - 1)), 1 << (bits - 1), size=(3, 64))
    b = sp.pack_bits(codes, bits)
    assert b.shape == (3, 64 * bits // 8)
    for row in range(3):
        stream = [(int(b[row, i // 8]) >> (i % 8)) & 1 for i in range(64 * bits)]
        for t in range(64):
            v = sum(stream[bits * t + k] << k for k in range(bits))
            assert v == codes[row, t] & ((1 << bits) - 1)
    assert np.array_equal(sp.unpack_bits(b, bits), codes)


def test_anchor_error_falls_with_width_and_full_codes_agree():
    """The full reconstruction is the same for every split (the 8-bit code is
    recovered exactly); the Anchor-only error falls as the Anchor widens."""
    x = _pages(2, 7)
    xf = lo.bf16_to_f32(x).astype(np.float64)
    full = None
    errs = []
    for A in (2, 3, 4, 5, 6):
        a, r, m = sp.encode_pages_split(x, A, 100.0, EPS)
        f = sp.reconstruct_split(a, r, m, A, 100.0, EPS)
        if full is None:
            full = f
        assert np.array_equal(f, full)
        errs.append(bl.vnmse(sp.reconstruct_split(a, None, m, A, 100.0, EPS), xf, axis=1))
    assert all(errs[i] > errs[i + 1] for i in range(len(errs) - 1)), errs
