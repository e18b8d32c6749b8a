"""Pins of oracle/baselines.py (single-precision Lynx variants, uniform INT8 /
INT4, vNMSE) to closed forms, invariants and the pinned Lynx oracle."""
import numpy as np
import pytest

from oracle import baselines as bl
from oracle import lynx_oracle as lo
from progressive_kv_quantization_gb300 import inputs

EPS = 1e-6


def _bf16(x: np.ndarray) -> np.ndarray:
    """float32 values that are BF16-exact -> BF16 bits."""
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _pages(n, seed):
    return inputs.kv_pages_np(1, 256 * n, seed, inputs.outlier_pairs(1, seed))


@pytest.mark.parametrize("bits", [4, 8])
def test_uniform_ramp_is_exact(bits):
    """A row holding every level min + k S (k = 0 .. 2^b - 1, S = 0.5) encodes to
    k and reconstructs exactly; each row's extremes map to 0 and 2^b - 1."""
    L = 2 ** bits
    k = np.arange(256) % L
    row = -3.0 + 0.5 * k
    x = _bf16(np.tile(row, (1, 128, 1)))
    q, mn, sc = bl.uniform_encode(x, bits)
    assert np.all(sc == 0.5) and np.all(mn == -3.0)
    assert np.array_equal(q[0, 0], k.astype(np.uint8))
    assert np.array_equal(bl.uniform_decode(q, mn, sc)[0, 0], row)


@pytest.mark.parametrize("bits", [4, 8])
def test_uniform_error_within_half_a_step(bits):
    """Synthetic KV pages: every code in 0 .. 2^b - 1, |x_hat - x| <= S/2 (+ float32
    rounding of the quotient), the minimum and maximum of each row exact."""
    x = _pages(3, 5)
    q, mn, sc = bl.uniform_encode(x, bits)
    xf = lo.bf16_to_f32(x).astype(np.float64)
    xh = bl.uniform_decode(q, mn, sc)
    assert q.max() <= 2 ** bits - 1
    err = np.abs(xh - xf)
    bound = sc.astype(np.float64)[..., None] * (0.5 + 1e-6) + 1e-6 * np.abs(xf)
    assert np.all(err <= bound)
    rows = np.arange(xf.shape[1])
    for n in range(xf.shape[0]):
        i_min, i_max = xf[n].argmin(axis=1), xf[n].argmax(axis=1)
        assert np.all(q[n, rows, i_min] == 0) and np.all(q[n, rows, i_max] == 2 ** bits - 1)


def test_uniform_constant_row_is_exact():
    x = _bf16(np.full((1, 128, 256), 1.75, dtype=np.float32))
    q, mn, sc = bl.uniform_encode(x, 4)
    assert np.all(q == 0) and np.all(sc == 0)
    assert np.all(bl.uniform_decode(q, mn, sc) == 1.75)


def test_pack_codes4_order_and_roundtrip():
    c = np.array([[1, 2, 15, 0]], dtype=np.uint8)
    assert list(bl.pack_codes4(c)[0]) == [0x21, 0x0F]
    r = np.random.default_rng(0).integers(0, 16, (3, 8, 256), dtype=np.uint8)
    assert np.array_equal(bl.unpack_codes4(bl.pack_codes4(r)), r)


def test_lynx_int8_is_the_full_code():
    """The one-byte code shifted right by 4 (arithmetically) is the Anchor, and it
    reconstructs to the full-code values of the split stream."""
    x = _pages(2, 9)
    q8, meta = bl.lynx_int8_encode(x, 100.0, EPS)
    a, r, m = lo.encode_pages(x, 100.0, EPS)
    assert np.array_equal(m, meta)
    assert np.array_equal(q8.astype(np.int32) >> 4, lo.unpack_nibbles(a).astype(np.int32))
    full = lo.reconstruct(a, r, m, 100.0, EPS)
    assert np.allclose(bl.lynx_int8_decode(q8, meta, 100.0, EPS), full, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("alpha", [1.0, 100.0, 1e4])
def test_int4_compander_bins(alpha):
    """Every level k of the 7-level compander: its centre expander4(k) maps back
    to k, and values just inside either edge of its bin round to k."""
    k = np.arange(8, dtype=np.float64)
    c = bl.expander4(k, alpha)
    assert np.allclose(bl.compander4(c, alpha), k, atol=1e-12)
    lo_edge = bl.expander4(np.maximum(k - 0.5 + 1e-6, 0), alpha)
    hi_edge = bl.expander4(np.minimum(k + 0.5 - 1e-6, 7), alpha)
    assert np.array_equal(np.rint(bl.compander4(lo_edge, alpha)), k)
    assert np.array_equal(np.rint(bl.compander4(hi_edge, alpha)), k)
    assert bl.expander4(7, alpha) == pytest.approx(1.0, abs=1e-15)


def test_lynx_int4_two_level_row_closed_form():
    """A row alternating two values has x_f = -1 / +1 everywhere (chunk mean in
    the middle), so every code is the extreme level 7 and the row reconstructs
    to its two values (up to eps)."""
    row = np.where(np.arange(256) % 2 == 0, -2.0, 6.0)
    x = _bf16(np.tile(row, (1, 128, 1)))
    packed, meta = bl.lynx_int4_encode(x, 100.0, EPS)
    q = lo.unpack_nibbles(packed)
    assert np.all(q[0, :, 0::2] == -8) and np.all(q[0, :, 1::2] == 7)
    xh = bl.lynx_int4_decode(packed, meta, 100.0, EPS)
    assert np.allclose(xh[0], np.tile(row, (128, 1)), atol=1e-4)


def test_lynx_int4_error_bound_and_ordering():
    """Each code is within half a level of the companded |x_f| (the rounding),
    codes lie in [-8, 7], and the 7-level reconstruction errs more than the
    127-level (full 8-bit) one."""
    x = _pages(2, 13)
    packed, meta, Y = bl.lynx_int4_encode(x, 100.0, EPS, return_y=True)
    q = lo.unpack_nibbles(packed).astype(np.int32)
    I4 = np.where(q < 0, -q - 1, q)
    assert q.min() >= -8 and q.max() <= 7
    assert np.all(np.abs(I4 - Y) <= 0.5 + 1e-9)
    xf = lo.bf16_to_f32(x).astype(np.float64)
    a, r, m = lo.encode_pages(x, 100.0, EPS)
    e4 = bl.vnmse(bl.lynx_int4_decode(packed, meta, 100.0, EPS), xf, axis=1)
    e8 = bl.vnmse(lo.reconstruct(a, r, m, 100.0, EPS), xf, axis=1)
    assert e4 > e8


def test_vnmse_closed_forms():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((5, 128, 7))
    assert bl.vnmse(v, v, axis=1) == 0.0
    assert bl.vnmse(1.1 * v, v, axis=1) == pytest.approx(0.01, rel=1e-12)
    w = v.copy()
    w[:, 0, :] = 0.0                       # one channel dropped: its energy share
    share = np.mean(v[:, 0, :] ** 2 / np.sum(v ** 2, axis=1))
    assert bl.vnmse(w, v, axis=1) == pytest.approx(share, rel=1e-12)
