"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties the oracle to something other than itself: values printed on
the pages (tests/golden/*.json), closed forms, exact special cases and
error bounds.  No GPU is needed.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import lynx_oracle as lo
from progressive_kv_quantization_gb300 import inputs

GOLD = os.path.join(os.path.dirname(__file__), "golden")
EPS = np.float32(1e-6)


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _bf16(x):
    return inputs.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


# ---------------------------------------------------------------- worked example

def test_worked_example_stage3_matches_printed_values():
    g = _gold("worked_example.json")
    a = g["alpha"]
    xf = (g["x_before_centering"] - g["mu"]) / g["sigma"]
    assert abs(xf - g["x_final_printed"]) < 5e-4
    # Eq. (13)'s printed pieces: 1 + 255*0.673, ln of it, ln 256
    assert abs(1 + a * g["x_final_printed"] - g["eq13_argument_printed"]) < 0.1
    assert abs(math.log(g["eq13_argument_printed"]) - g["eq13_ln_numerator_printed"]) < 1e-3
    assert abs(math.log(1 + a) - g["eq13_ln_denominator_printed"]) < 1e-3
    Y = float(lo.compander(xf, a))
    assert abs(Y - g["Y_printed"]) < 0.1
    Yq, I, S = lo.quantise(np.array([xf], dtype=np.float32), np.float32(a))
    assert int(I[0]) == g["I"] and int(S[0]) == g["sign"]


def test_worked_example_stage4_literal_lines_match_printed_values():
    g = _gold("worked_example.json")
    out = lo.split_stream_literal(np.array([g["I"]]), np.array([g["sign"]]))
    p = g["stage4_printed"]
    assert int(out["I_bias"][0]) == p["I_bias"]
    assert int(out["V_mag"][0]) == p["V_mag"]
    assert int(out["V_recon"][0]) == p["V_recon"]
    assert int(out["Q_res"][0]) == p["V_res"] == p["Q_res"]
    assert int(out["Q_anc"][0]) == p["Q_anc"]
    # full reconstruction index printed in Eq. (15): V_recon - Q_res
    assert int(out["V_recon"][0] - out["Q_res"][0]) == g["I_full_printed"]


def test_worked_example_reading_b_and_reconstruction():
    g = _gold("worked_example.json")
    q_anc, q_res = lo.split_stream(np.array([g["I"]]), np.array([g["sign"]]))
    # reading B: V = 118 >> 4 = 7, anchor = 7, residual = 16*7 + 7 - 118 = 1
    assert int(q_anc[0]) == 7 and int(q_res[0]) == 1
    # the full code reconstructs the same index as the printed Eq. (15)
    assert 16 * 7 + 7 - int(q_res[0]) == g["I_full_printed"]
    # the page's claim: full reconstruction within 1% of |x_final|
    full = float(lo.expander(g["I_full_printed"], g["alpha"]))
    assert abs(full - g["x_final_printed"]) / g["x_final_printed"] < g["full_reconstruction_relative_error_below"]
    # the printed 0.729 / 0.668 / 187 do not follow from Eq. (14)'s own formula
    bad = g["printed_inconsistent"]
    assert abs(256 ** (112 / 127) - bad["intermediate_256_pow_0_882"]) > 40
    assert abs(float(lo.expander(112, g["alpha"])) - bad["anchor_only_abs_x_hat"]) > 0.1
    assert abs(full - bad["full_abs_x_hat"]) > 4e-3


# ---------------------------------------------------------------- compander

@pytest.mark.parametrize("alpha", [1.0, 100.0, 255.0, 1000.0])
def test_compander_inverse_closed_form(alpha):
    x = np.linspace(0.0, 1.0, 20001)
    y = lo.compander(x, alpha)
    assert np.max(np.abs(lo.expander(y, alpha) - x)) < 1e-12
    yy = np.linspace(0.0, 127.0, 1271)
    assert np.max(np.abs(lo.compander(lo.expander(yy, alpha), alpha) - yy)) < 1e-9
    assert float(lo.compander(0.0, alpha)) == 0.0
    assert abs(float(lo.compander(1.0, alpha)) - 127.0) < 1e-12
    assert np.all(np.diff(y) > 0)
    # slope at 0 of 127 ln(1 + a x)/ln(1 + a) is 127 a / ln(1 + a)
    h = 1e-9
    slope = (float(lo.compander(h, alpha)) - 0.0) / h
    assert abs(slope - 127 * alpha / math.log1p(alpha)) / slope < 1e-6
    # fp32 round trip (the north-star's 1e-6 identity check)
    x32 = x.astype(np.float32)
    back = lo.expander(lo.compander(x32, alpha), alpha).astype(np.float32)
    assert np.max(np.abs(back - x32)) < 1e-6


@pytest.mark.parametrize("alpha", [100.0, 255.0])
def test_quantise_every_bin(alpha):
    a32 = np.float32(alpha)
    for k in range(128):
        centre = np.float32(lo.expander(k, alpha))
        _, I, S = lo.quantise(np.array([centre, -centre], dtype=np.float32), a32)
        assert list(I) == [k, k]
        assert int(S[0]) == 1 and int(S[1]) == (-1 if centre > 0 else 1)
        if k < 127:
            edge = lo.expander(k + 0.5, alpha)
            above = np.float32(edge * (1 + 1e-6))
            below = np.float32(edge * (1 - 1e-6))
            _, I2, _ = lo.quantise(np.array([below, above], dtype=np.float32), a32)
            assert list(I2) == [k, k + 1]


# ---------------------------------------------------------------- stage 4

def test_sign_aware_map_printed_cases():
    g = _gold("printed_values.json")["sign_aware_map"]
    for c in g["cases"]:
        I = np.array([c["V_mag"] << 4])
        q_anc, _ = lo.split_stream(I, np.array([c["S"]]))
        assert int(q_anc[0]) == c["Q_anc"]


def test_split_stream_identities_all_codes():
    I = np.tile(np.arange(128), 2)
    S = np.repeat([1, -1], 128)
    q_anc, q_res = lo.split_stream(I, S)
    q8 = np.where(S > 0, I, -I - 1)              # signed 8-bit code
    assert q8.min() == -128 and q8.max() == 127
    assert np.array_equal(q_anc.astype(np.int32), q8 >> 4)   # anchor = full code >> 4
    V = I >> 4
    assert np.array_equal(16 * V + 7 - q_res.astype(np.int32), I)
    assert q_anc.min() == -8 and q_anc.max() == 7
    assert q_res.min() == -8 and q_res.max() == 7
    # Stage 4 as printed needs a ninth magnitude level once I + 7 >= 128
    lit = lo.split_stream_literal(I, S)
    assert np.array_equal(lit["V_mag"] == 8, I >= 121)
    assert lit["Q_anc"].min() == -9 and lit["Q_anc"].max() == 8


def test_pack_nibble_order_and_roundtrip():
    q = np.array([[1, 2, -1, -8, 7, 0]])
    b = lo.pack_nibbles(q)
    assert list(b[0]) == [0x21, 0x8F, 0x07]        # low nibble = even token
    assert np.array_equal(lo.unpack_nibbles(b), q)
    r = np.random.default_rng(1).integers(-8, 8, size=(3, 256))
    assert np.array_equal(lo.unpack_nibbles(lo.pack_nibbles(r)), r)


# ---------------------------------------------------------------- stages 1-2

def _pages(seed=0):
    return inputs.kv_pages_np(1, 256 * 4, seed, inputs.outlier_pairs(1, seed, count=4))


def test_normalisation_invariants():
    x_bits = _pages()
    st = lo.run_stages(x_bits, 100.0, EPS)
    x = lo.bf16_to_f32(x_bits)
    assert st.xn.min() >= 0.0 and st.xn.max() <= 1.0
    n, H, P = x.shape
    rows = np.arange(n * H)
    xn = st.xn.reshape(n * H, P)
    xr = x.reshape(n * H, P)
    assert np.all(xn[rows, xr.argmin(axis=1)] == 0.0)
    assert np.all(xn[rows, xr.argmax(axis=1)] > 1.0 - 1e-5)
    assert np.all(st.gmin == x.min(axis=2))                    # gamma_min is exact
    assert np.all(np.abs(st.xfinal) <= 1.0)
    # one element per chunk attains sigma / (sigma + eps)
    top = np.abs(st.xfinal).max(axis=3)
    assert np.all(top == st.sigma / (st.sigma + EPS))
    # the chunk mean is within the float32 error bound of the exact mean
    exact = st.xn.reshape(n, H, P // 32, 32).astype(np.float64).mean(axis=3)
    assert np.max(np.abs(st.mu - exact)) <= 32 * 2.0 ** -24


def test_constant_row_encodes_to_zero_and_reconstructs():
    x = np.zeros((1, 128, 256), dtype=np.float32)
    x[0] = np.linspace(-3, 3, 256, dtype=np.float32)[None, :]
    x[0, 5, :] = 1.5                                       # one constant channel
    bits = _bf16(x)
    anc, res, meta, st = lo.encode_pages(bits, 100.0, EPS, return_stages=True)
    assert st.gscale[0, 5] == 0.0 and np.all(st.mu[0, 5] == 0) and np.all(st.sigma[0, 5] == 0)
    assert np.all(st.I[0, 5] == 0) and np.all(st.S[0, 5] == 1)
    assert np.all(anc[0, 5] == 0x00) and np.all(res[0, 5] == 0x77)   # residual = 7 per nibble
    for r in (None, res):
        xh = lo.reconstruct(anc, r, meta, 100.0, EPS)
        assert np.max(np.abs(xh[0, 5] - 1.5)) < 1e-9


def test_two_level_row_closed_form():
    a, b = np.float32(-2.0), np.float32(6.0)
    x = np.full((1, 128, 256), a, dtype=np.float32)
    x[0, :, 1::2] = b                                      # alternate a, b
    st = lo.run_stages(_bf16(x), 100.0, EPS)
    top = np.float32(8.0) / (np.float32(8.0) + EPS)      # x_norm of the b tokens
    assert np.all(st.xn[0, :, 1::2] == top) and np.all(st.xn[0, :, 0::2] == 0)
    # 16 zeros and 16 tops summed in float32: within the summation error bound of top/2
    assert np.max(np.abs(st.mu.astype(np.float64) - float(top) / 2)) <= 16 * 2.0 ** -24
    assert np.all(st.I == 127)                            # |x_final| = 1 - O(eps)
    q_anc, q_res = lo.split_stream(st.I, st.S)
    assert np.all(q_anc[0, :, 0::2] == -8) and np.all(q_anc[0, :, 1::2] == 7)
    assert np.all(q_res == -8)


def test_ramp_row_closed_form_codes():
    alpha = 100.0
    x = np.tile(np.arange(256, dtype=np.float32), (1, 128, 1))  # integers: exact in BF16
    st = lo.run_stages(_bf16(x), alpha, EPS)
    # closed form: x_norm = t/255, chunk c has mean (32c + 15.5)/255 and max deviation 15.5/255,
    # so x_final = (j - 15.5)/15.5 for the j-th token of every chunk
    j = np.arange(256) % 32
    sig = 15.5 / 255.0
    xf_exact = (j - 15.5) / 15.5 * sig / (sig + 1e-6)
    assert np.max(np.abs(st.mu[0, 0] - (32 * np.arange(8) + 15.5) / 255.0)) < 2e-6
    assert np.max(np.abs(st.sigma[0, 0] - 15.5 / 255.0)) < 2e-6
    # float32 bound: the mean of 32 values near 1 carries up to 32 ulp(1), amplified by 1/sigma
    assert np.max(np.abs(st.xfinal[0, 0].reshape(-1) - xf_exact)) < 33 * 2.0 ** -24 / sig
    Y = lo.compander(np.abs(xf_exact), alpha)
    I_exact = np.rint(Y)
    clear = np.abs(Y - np.floor(Y) - 0.5) > 0.05          # not near a rounding edge
    assert clear.sum() > 200
    assert np.array_equal(st.I[0, 0][clear], I_exact[clear])
    assert np.array_equal(st.S[0, 0], np.where(j < 16, -1, 1))


# ---------------------------------------------------------------- reconstruction

def _step_bounds(I, alpha, anchor):
    """Largest |x_final - x_hat_final| allowed by the code: half a code step for
    the full code, the anchor bin's extent for the anchor alone."""
    if anchor:
        V = I >> 4
        c = 16 * V + 7
        lo_edge = np.maximum(16 * V - 0.5, 0.0)
        hi_edge = np.minimum(16 * V + 15.5, 127.0)
    else:
        c = I
        lo_edge = np.maximum(I - 0.5, 0.0)
        hi_edge = np.minimum(I + 0.5, 127.0)
    e = lambda y: lo.expander(y, alpha)
    return np.maximum(e(hi_edge) - e(c), e(c) - e(lo_edge))


@pytest.mark.parametrize("alpha", [100.0, 255.0])
def test_reconstruction_error_bounded_by_code_step(alpha):
    x_bits = _pages(3)
    anc, res, meta, st = lo.encode_pages(x_bits, alpha, EPS, return_stages=True)
    x = lo.bf16_to_f32(x_bits).astype(np.float64)
    n, H, P = x.shape
    ds = np.repeat((st.sigma + EPS).astype(np.float64), 32, axis=2)
    dg = (st.gscale + EPS).astype(np.float64)[..., None]
    slack = 8 * 2.0 ** -24 * (np.abs(x) + np.abs(st.gmin)[..., None] + dg * (2 + ds))
    for anchor, r in ((True, None), (False, res)):
        xh = lo.reconstruct(anc, r, meta, alpha, EPS)
        bound = dg * ds * _step_bounds(st.I, alpha, anchor) + slack
        assert np.all(np.abs(xh - x) <= bound)


def test_anchor_error_not_below_full_code_error():
    x_bits = _pages(4)
    anc, res, meta, st = lo.encode_pages(x_bits, 100.0, EPS, return_stages=True)
    # code domain, per element: I = Round(Y) is the nearest index to Y
    i_anc = 16 * (st.I >> 4) + 7
    assert np.all(np.abs(st.Y - i_anc) >= np.abs(st.Y - st.I))
    # value domain, per chunk: summed squared error
    x = lo.bf16_to_f32(x_bits).astype(np.float64)
    e_anc = (lo.reconstruct(anc, None, meta, 100.0, EPS) - x) ** 2
    e_full = (lo.reconstruct(anc, res, meta, 100.0, EPS) - x) ** 2
    n, H, P = x.shape
    sa = e_anc.reshape(n, H, 8, 32).sum(axis=3)
    sf = e_full.reshape(n, H, 8, 32).sum(axis=3)
    assert np.all(sa >= sf)


# ---------------------------------------------------------------- sizes

def test_kv_size_closed_form():
    g = _gold("printed_values.json")["kv_size"]
    size = g["K_factor"] * g["seq_len"] * g["n_kv_heads"] * g["head_dim"] * g["n_layers"] * g["bytes_per_element"]
    assert size == 25_232_932_864
    assert round(size / 2 ** 30, 1) == g["printed_GB"]           # the page's GB is GiB
    w = inputs.QWEN235B_CACHE
    assert w.bf16_bytes == size
    assert 2 * w.n_layers * w.pages_per_tensor_layer * 128 * 256 * 2 == size
    assert inputs.QWEN32B_CACHE.bf16_bytes == 4_294_967_296


def test_metadata_size_printed():
    g = _gold("printed_values.json")["metadata_overhead"]
    n = lo.meta_size(g["H"], g["P"], g["C"])
    assert n == g["scalars"]
    assert round(n * 4 / 1024) == g["printed_KB_fp32"]
    assert round(n * 4 / (g["H"] * g["P"] * 2), 2) == g["printed_overhead_fraction"]


# ---------------------------------------------------------------- partial pages
def _partial_pages(n, seed):
    out = inputs.outlier_pairs(1, seed)
    return inputs.kv_pages_np(1, 256 * n, seed, out)


def test_partial_rule_with_full_pages_is_the_full_page_rule():
    x = _partial_pages(3, 31)
    full = lo.encode_pages(x, 100.0, 1e-6)
    part = lo.encode_pages(x, 100.0, 1e-6, valid=np.full(3, 256))
    for a, b in zip(full, part):
        assert np.array_equal(a, b)


def test_partial_page_ignores_its_padding():
    """Whatever the padding holds (other values, huge values, NaN or Inf bits),
    the valid tokens' codes and every metadata value stay the same, and padding
    tokens get code 0 with a positive sign (anchor 0, residual 7)."""
    rng = np.random.default_rng(7)
    x = _partial_pages(4, 32)
    valid = np.array([1, 77, 200, 255])
    ref = lo.encode_pages(x, 100.0, 1e-6, valid=valid)
    for fill in ("random", "huge", "nonfinite"):
        y = x.copy()
        for n, v in enumerate(valid):
            if fill == "random":
                y[n, :, v:] = rng.integers(0, 1 << 16, y[n, :, v:].shape, dtype=np.uint16) & 0x7F7F
            elif fill == "huge":
                y[n, :, v:] = 0x7F00                      # 2^127
            else:
                y[n, :, v:] = np.where(rng.random(y[n, :, v:].shape) < 0.5, 0x7FC0, 0xFF80)
        got = lo.encode_pages(y, 100.0, 1e-6, valid=valid)
        for a, b in zip(ref, got):
            assert np.array_equal(a, b)
    qa = lo.unpack_nibbles(ref[0])
    qr = lo.unpack_nibbles(ref[1])
    for n, v in enumerate(valid):
        assert np.all(qa[n, :, v:] == 0) and np.all(qr[n, :, v:] == 7)


def test_partial_page_whole_chunks_match_a_full_page_with_neutral_padding():
    """If the invalid tokens form whole chunks and are filled with the row's valid
    minimum (so that min and max do not change), the valid chunks' codes and
    statistics equal those of the full-page encoding of the filled page."""
    x = _partial_pages(1, 33)
    v = 160                                           # chunks 0-4 valid, 5-7 invalid
    xf = lo.bf16_to_f32(x)
    y = x.copy()
    rowmin = np.argmin(xf[0, :, :v], axis=1)
    for c in range(128):
        y[0, c, v:] = x[0, c, rowmin[c]]
    a_p, r_p, m_p = lo.encode_pages(x, 100.0, 1e-6, valid=[v])
    a_f, r_f, m_f = lo.encode_pages(y, 100.0, 1e-6)
    assert np.array_equal(a_p[0, :, :v // 2], a_f[0, :, :v // 2])
    assert np.array_equal(r_p[0, :, :v // 2], r_f[0, :, :v // 2])
    gp, sp, mup, sgp = lo.unpack_meta(m_p, 128, 256, 32)
    gf, sf, muf, sgf = lo.unpack_meta(m_f, 128, 256, 32)
    assert np.array_equal(gp, gf) and np.array_equal(sp, sf)
    assert np.array_equal(mup[..., :5], muf[..., :5]) and np.array_equal(sgp[..., :5], sgf[..., :5])
    assert np.all(mup[..., 5:] == 0) and np.all(sgp[..., 5:] == 0)


def test_partial_page_statistics_brute_force():
    """gamma_min / gamma_scale are the min and the float32 range of the valid
    tokens; a partly valid chunk's mu is within float32 summation error of the
    float64 mean of its valid x_n and its sigma is the largest deviation among
    them; a page with no valid token has all-zero metadata."""
    x = _partial_pages(2, 34)
    valid = np.array([77, 0])
    st = lo.run_stages(x, 100.0, 1e-6, valid=valid)
    xf = lo.bf16_to_f32(x).astype(np.float64)
    v = 77
    assert np.array_equal(st.gmin[0], xf[0, :, :v].min(axis=1).astype(np.float32))
    assert np.array_equal(st.gscale[0], (xf[0, :, :v].max(axis=1) - xf[0, :, :v].min(axis=1)).astype(np.float32))
    xn = st.xn[0].astype(np.float64)                  # [128, 256]
    for c in range(3):                                # chunk 2 holds 13 valid tokens
        lo_t, hi_t = 32 * c, min(32 * c + 32, v)
        ref_mu = xn[:, lo_t:hi_t].mean(axis=1)
        assert np.all(np.abs(st.mu[0, :, c] - ref_mu) <= 32 * 2.0 ** -24 * np.maximum(1.0, np.abs(ref_mu)))
        dev = np.abs(xn[:, lo_t:hi_t] - st.mu[0, :, c:c + 1].astype(np.float64))
        assert np.all(np.abs(st.sigma[0, :, c] - dev.max(axis=1)) <= 2.0 ** -23)
    assert np.all(st.mu[0, :, 3:] == 0) and np.all(st.sigma[0, :, 3:] == 0)
    assert np.all(st.gmin[1] == 0) and np.all(st.gscale[1] == 0)
    assert np.all(st.mu[1] == 0) and np.all(st.sigma[1] == 0) and np.all(st.I[1] == 0)


def test_token_major_pages_brute_force():
    """pages_from_tokens: every element of a 300-token, 2-head token-major block
    (with two extra columns per row) lands at page h * n_pp + t // 256, channel
    c, position t % 256; padding is zero and the valid counts are 256 and 44."""
    rng = np.random.default_rng(5)
    n_tokens, n_heads = 300, 2
    x = rng.integers(0, 1 << 16, size=(n_tokens, n_heads * 128 + 2), dtype=np.uint16)
    pages, valid = lo.pages_from_tokens(x, n_heads)
    assert pages.shape == (4, 128, 256) and list(valid) == [256, 44, 256, 44]
    for t in range(n_tokens):
        for h in range(n_heads):
            assert np.array_equal(pages[h * 2 + t // 256, :, t % 256], x[t, h * 128:(h + 1) * 128])
    assert not pages[1, :, 44:].any() and not pages[3, :, 44:].any()


def test_token_major_encode_is_the_page_encode_of_the_same_tokens():
    """A head whose tokens fill whole pages encodes, through the token-major
    entry, exactly as those pages do through the page encoder (the layout
    changes where the values come from, nothing else), and a ragged last page
    encodes as a partial page of its valid tokens."""
    x_pages = inputs.kv_pages_np(1, 768, 33, inputs.outlier_pairs(1, 33))   # 3 pages of one head
    # token-major rows of that head: token t = page t // 256, position t % 256
    x_tm = np.concatenate([x_pages[j].T for j in range(3)], axis=0)[:612]
    a, r, m = lo.encode_tokens(x_tm, 1, 100.0, 1e-6)
    a2, r2, m2 = lo.encode_pages(x_pages[:2], 100.0, 1e-6)
    assert np.array_equal(a[:2], a2) and np.array_equal(r[:2], r2) and np.array_equal(m[:2], m2)
    a3, r3, m3 = lo.encode_pages(x_pages[2:], 100.0, 1e-6, valid=np.array([100]))
    assert np.array_equal(a[2:], a3) and np.array_equal(r[2:], r3) and np.array_equal(m[2:], m3)
