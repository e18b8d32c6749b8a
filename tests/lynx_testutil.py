"""Shared helpers for the parity tests: comparison rules derived from the code
definition and the arithmetic (no GPU code here)."""
from __future__ import annotations

import numpy as np

from oracle import lynx_oracle as lo

EPS = np.float32(1e-6)
CODE_EDGE = 1e-5          # codes may differ by 1 only where the oracle's Y is this close to k + 1/2
CODE_FRACTION = 1e-4      # and at most this fraction of codes may differ
ATTN_TOL = 2e-3           # |gpu - oracle| <= ATTN_TOL * max(1, |oracle|)


def full_codes(anchor: np.ndarray, residual: np.ndarray) -> np.ndarray:
    """Signed 8-bit codes (S>0 ? I : -I-1) recovered from the two packed planes."""
    qa = lo.unpack_nibbles(anchor).astype(np.int32)
    qr = lo.unpack_nibbles(residual).astype(np.int32)
    S = np.where(qa < 0, -1, 1)
    V = np.where(S > 0, qa, -qa - 1)
    I = 16 * V + 7 - qr
    return np.where(S > 0, I, -I - 1)


# (differing codes, codes compared) of every check_codes call of the session,
# reported at the end of the run (conftest's terminal summary)
CODE_TALLY = []


def check_codes(gpu_anchor, gpu_res, ora_anchor, ora_res, Y):
    """Codes must be bit-exact except +-1 where the oracle's float64 Y is within
    CODE_EDGE of a rounding edge; returns the fraction of differing codes."""
    g = full_codes(np.asarray(gpu_anchor), np.asarray(gpu_res))
    o = full_codes(np.asarray(ora_anchor), np.asarray(ora_res))
    diff = g != o
    n = int(diff.sum())
    if n:
        Yd = np.asarray(Y)[diff]
        near = np.abs(Yd - np.floor(Yd) - 0.5) < CODE_EDGE
        # a +-1 step of the magnitude across zero turns code 0 into -1, so compare magnitudes
        mag = lambda q: np.where(q < 0, -q - 1, q)
        step = np.abs(mag(g[diff]) - mag(o[diff]))
        assert np.all(near), f"{n} codes differ, {int((~near).sum())} of them away from a rounding edge"
        assert np.all(step <= 1)
    frac = n / g.size
    CODE_TALLY.append((n, g.size))
    assert frac < CODE_FRACTION, f"differing-code fraction {frac}"
    return frac


def check_meta(gpu_meta, ora_meta):
    g = np.asarray(gpu_meta, dtype=np.float64)
    o = np.asarray(ora_meta, dtype=np.float64)
    assert np.all(np.abs(g - o) <= 1e-6 * np.abs(o) + 1e-7), "metadata differs beyond 1e-6 relative"
    return float(np.mean(g == o))


def recon_bound(meta, H=128, P=256, C=32):
    """Per-element bound on |float32 reconstruction - float64 reconstruction|.

    The float32 path rounds the table value S*l (|l| <= 1), the inner fused
    multiply-add t = l*ds + mu and the outer one x = t*dg + gamma_min once each
    (relative 2^-24); ds = sigma+eps and dg = gamma_scale+eps are the same
    float32 sums on both sides.  That error is at most
    2^-24 (3 ds dg + 2 |mu| dg + |gamma_min|); the bound takes 2^-21 per term.
    """
    gmin, gscale, mu, sigma = lo.unpack_meta(meta, H, P, C)
    ds = np.repeat((sigma + EPS).astype(np.float64), C, axis=2)
    dg = (gscale + EPS).astype(np.float64)[..., None]
    mu_e = np.repeat(np.abs(mu.astype(np.float64)), C, axis=2)
    return 2.0 ** -21 * (ds * dg + mu_e * dg + np.abs(gmin.astype(np.float64))[..., None])


def bf16_ulp(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def check_recon(gpu, oracle64, bound, is_bf16):
    """float32 output: within ``bound`` of the float64 value.  BF16 output: the
    float32 result rounded to BF16, i.e. within half a BF16 ulp plus ``bound``."""
    g = np.asarray(gpu, dtype=np.float64)
    lim = bound
    if is_bf16:
        lim = lim + 0.5 * bf16_ulp(np.maximum(np.abs(g), np.abs(oracle64)))
    err = np.abs(g - oracle64)
    bad = err > lim
    assert not bad.any(), f"{int(bad.sum())} elements beyond the bound (max err {err.max()})"


def check_attention(o_gpu, lse_gpu, o_ref, lse_ref, mask=None):
    og = np.asarray(o_gpu, dtype=np.float64)
    lg = np.asarray(lse_gpu, dtype=np.float64)
    if mask is not None:
        og, lg, o_ref, lse_ref = og[mask], lg[mask], o_ref[mask], lse_ref[mask]
    eo = np.abs(og - o_ref) / np.maximum(1.0, np.abs(o_ref))
    fin = np.isfinite(lse_ref)
    el = np.abs(lg[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
    assert np.all(np.isneginf(lg[~fin]))
    assert eo.max() <= ATTN_TOL, f"attention output error {eo.max()}"
    assert el.size == 0 or el.max() <= ATTN_TOL, f"lse error {el.max()}"
    return float(eo.max()), float(el.max() if el.size else 0.0)
