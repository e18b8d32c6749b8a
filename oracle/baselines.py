"""Plain CPU oracle of the single-precision Lynx variants and of the uniform
INT8 / INT4 KV quantisers the Lynx paper compares against, and of the error
measures of the paper's Table 3.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  The
library never calls it and shares no code, tables or constants with the CUDA
path.  Every function is pinned (tests/test_oracle_baselines.py) to closed
forms, invariants or the pinned Lynx oracle.

Sources (cited by page title and section; no code is taken from them):
  [paper] "Lynx: Progressive Speculative Quantization for accelerating KV
          Transfer in Long-Context Inference": §2.3 "Standard & Grouped
          Quantization" (Q(X) = round(X/S + Z) with S from the range
          [x_min, x_max], independent scales per block); §6.1 "Baselines" and
          "Lynx's configurations" (uniform INT8 and INT4; Lynx-INT4 and
          Lynx-INT8 quantise with the hierarchical algorithm of §4.1 at a
          single precision, without the split stream); §6.2, Table 3 (vNMSE of
          each method).

Readings of the pages (all listed in the design notes):
  * Uniform INT-b.  A block is one channel row of a page (the 256 tokens over
    which Lynx takes gamma_min / gamma_scale).  S = (max - min) / (2^b - 1)
    and the zero point is kept as the float -min/S, i.e. Q = round((x - min) / S)
    in 0 .. 2^b - 1 and x_hat = min + Q * S (the same affine family as
    round(X/S + Z); a constant row, S = 0, gets Q = 0 and is exact).  Float32
    arithmetic, one correctly rounded operation per step, round half to even.
    INT4 codes are packed two per byte, low nibble = even token.
  * Lynx-INT8.  Algorithm 1's 8-bit code, sign and 7-bit magnitude I, as one
    signed byte q8 = S > 0 ? I : -I - 1 (whose arithmetic shift by 4 is the
    Anchor), with Lynx's metadata; its values are those of Lynx's full codes.
  * Lynx-INT4.  Algorithm 1 with 2^3 - 1 = 7 magnitude levels:
    I4 = round(7 ln(1 + alpha |x_f|) / ln(1 + alpha)), stored as the sign-aware
    4-bit code S > 0 ? I4 : -I4 - 1 (two per byte, as the Anchor), with Lynx's
    metadata; x_hat_f = S l4(I4), l4(y) = ((1 + alpha)^(y/7) - 1) / alpha.
  * vNMSE (Table 3 names it without a formula): for a set of vectors v with
    estimates v_hat, the mean over the vectors of ||v_hat - v||^2 / ||v||^2.
    For KV the vectors are one head's 128 channels at one token.
"""
from __future__ import annotations

import numpy as np

from oracle import lynx_oracle as lo

INT4_LEVELS = 7


# ------------------------------------------------------------------ uniform INT-b

def uniform_encode(x_bits: np.ndarray, bits: int):
    """Uniform INT-b on BF16 pages [N, H, P]: returns (codes uint8 [N, H, P]
    (one code per token, 0 .. 2^b - 1), row_min float32 [N, H], scale float32
    [N, H])."""
    assert bits in (4, 8)
    x = lo.bf16_to_f32(x_bits)
    mn = x.min(axis=2)
    mx = x.max(axis=2)
    levels = np.float32(2 ** bits - 1)
    scale = (mx - mn) / levels                          # float32, correctly rounded
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (x - mn[..., None]) / scale[..., None]      # float32
    q = np.where(scale[..., None] > 0, np.rint(t), 0.0)
    q = np.clip(q, 0, 2 ** bits - 1).astype(np.uint8)
    return q, mn.astype(np.float32), scale.astype(np.float32)


def uniform_decode(codes: np.ndarray, row_min: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """x_hat = min + Q * S, in float64, [N, H, P]."""
    return row_min.astype(np.float64)[..., None] + codes.astype(np.float64) * scale.astype(np.float64)[..., None]


def pack_codes4(codes: np.ndarray) -> np.ndarray:
    """Unsigned 4-bit codes [..., P] -> bytes [..., P/2], low nibble = even token."""
    c = codes.astype(np.uint8)
    return (c[..., 0::2] & 0x0F) | ((c[..., 1::2] & 0x0F) << 4)


def unpack_codes4(b: np.ndarray) -> np.ndarray:
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0x0F
    out[..., 1::2] = b >> 4
    return out


# ------------------------------------------------------------------ Lynx-INT8

def lynx_int8_encode(x_bits: np.ndarray, alpha, eps, C: int = 32):
    """Algorithm 1's 8-bit code as one signed byte per token: (q8 int8 [N, H, P],
    meta float32 [N, 2304]) with Lynx's metadata layout."""
    st = lo.run_stages(x_bits, alpha, eps, C)
    q8 = np.where(st.S > 0, st.I, -st.I - 1).astype(np.int8)
    return q8, lo.pack_meta(st.gmin, st.gscale, st.mu, st.sigma)


def lynx_int8_decode(q8: np.ndarray, meta: np.ndarray, alpha, eps, H: int = 128, P: int = 256,
                     C: int = 32) -> np.ndarray:
    """x_f = S l(I), then the two affine steps of the reconstruction (float64)."""
    q = q8.astype(np.int32)
    S = np.where(q < 0, -1, 1)
    I = np.where(q < 0, -q - 1, q)
    xf = S * lo.expander(I, np.float32(alpha))
    return _affine(xf, meta, eps, H, P, C)


# ------------------------------------------------------------------ Lynx-INT4

def compander4(x_abs, alpha):
    """The alpha-law of Eq. (3) scaled to 7 levels, float64."""
    a = np.float64(alpha)
    return np.log1p(a * np.asarray(x_abs, dtype=np.float64)) / np.log1p(a) * INT4_LEVELS


def expander4(y, alpha):
    """Inverse of compander4: ((1 + alpha)^(y/7) - 1) / alpha, float64."""
    a = np.float64(alpha)
    return (np.power(1.0 + a, np.asarray(y, dtype=np.float64) / INT4_LEVELS) - 1.0) / a


def lynx_int4_encode(x_bits: np.ndarray, alpha, eps, C: int = 32, return_y: bool = False):
    """Stages 1-2 of Algorithm 1, then 7-level companded codes: (packed uint8
    [N, H, P/2] of S > 0 ? I4 : -I4 - 1, meta float32 [N, 2304]); with
    return_y also the float64 Y4 = compander4(|x_f|) [N, H, P]."""
    x = lo.bf16_to_f32(x_bits)
    N, H, P = x.shape
    gmin, gscale, xn, mu, xcent, sigma, xfinal = lo.normalise(x, C, eps)
    xf = xfinal.reshape(N, H, P)
    Y = compander4(np.abs(xf).astype(np.float64), np.float32(alpha))
    I4 = np.rint(Y).astype(np.int32)
    S = np.where(xf < 0, -1, 1)
    q4 = np.where(S > 0, I4, -I4 - 1).astype(np.int8)
    packed = lo.pack_nibbles(q4)
    meta = lo.pack_meta(gmin, gscale, mu, sigma)
    return (packed, meta, Y) if return_y else (packed, meta)


def lynx_int4_decode(packed: np.ndarray, meta: np.ndarray, alpha, eps, H: int = 128, P: int = 256,
                     C: int = 32) -> np.ndarray:
    q = lo.unpack_nibbles(packed).astype(np.int32)
    S = np.where(q < 0, -1, 1)
    I4 = np.where(q < 0, -q - 1, q)
    xf = S * expander4(I4, np.float32(alpha))
    return _affine(xf, meta, eps, H, P, C)


def _affine(xf, meta, eps, H, P, C):
    """x = (x_f (sigma + eps) + mu) (gamma_scale + eps) + gamma_min, float64."""
    N = xf.shape[0]
    gmin, gscale, mu, sigma = lo.unpack_meta(meta, H, P, C)
    e = np.float32(eps)
    xn = xf.reshape(N, H, P // C, C) * (sigma + e).astype(np.float64)[..., None] + mu.astype(np.float64)[..., None]
    return xn.reshape(N, H, P) * (gscale + e).astype(np.float64)[..., None] + gmin.astype(np.float64)[..., None]


# ------------------------------------------------------------------ error measure

def vnmse(v_hat: np.ndarray, v: np.ndarray, axis: int = -1) -> float:
    """Mean over the vectors (along ``axis``) of ||v_hat - v||^2 / ||v||^2."""
    v = np.asarray(v, dtype=np.float64)
    d = np.asarray(v_hat, dtype=np.float64) - v
    return float(np.mean(np.sum(d * d, axis=axis) / np.sum(v * v, axis=axis)))
