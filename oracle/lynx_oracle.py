"""Plain CPU oracle of the Lynx hierarchical split-stream KV quantiser.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  The
library itself never calls it, and it shares no code, tables or constants with
the CUDA path.

Sources (cited by page title and section; no code is taken from them):
  [paper] "Lynx: Progressive Speculative Quantization for accelerating KV
          Transfer in Long-Context Inference", §4.1 "Hierarchical Quantization",
          Algorithm 1 and Eqs. (3)-(4); §5 "Implementation" (two 4-bit codes
          per byte).
  [notes] Zhongzhu Zhou, "Lynx 阅读笔记：渐进式推测量化加速解聚合 LLM 推理的
          KV 传输" (reading notes), Algorithm 1 restated as stages 1-4,
          Eqs. (7)-(9), and the worked example, Eqs. (12)-(15).

Precision.  Stages 1-2 (normalisation) are written in float32, one IEEE
operation per step of Algorithm 1, because the 8-bit code is decided from
their float32 result and the CUDA kernels take that decision from the same
float32 values.  The compander, the rounding decision and the whole of the
reconstruction are evaluated in float64.

Readings of the pages where they are silent, garbled or inconsistent (all of
them listed in the design notes):
  * Anchor/Residual split ("reading B").  As printed, Stage 4 of
    Algorithm 1 gives an anchor magnitude (I+7)>>4 in 0..8, i.e. 18 signed
    levels, which cannot be the 4-bit anchor the paper ships two per byte.
    Here the anchor magnitude is V = I >> 4 (the top 3 magnitude bits), the
    anchor is Stage 4's sign-aware two's-complement map of V, which equals the int8 code
    (S>0 ? I : -I-1) shifted right by 4, and the Round-Half-Down +7 bias moves
    to the reconstruction point V_recon = 16*V + 7, so the residual
    Q_res = V_recon - I is a centred signed 4-bit correction in [-8, 7].
    ``split_stream_literal`` keeps the printed lines for the worked example.
  * Sign source: Stage 3 prints Sign(X_view), but X_view lies in [0, 1]; the
    sign is taken from X_final, and zero counts as positive.
  * Mean over a chunk: the C values are summed left to right in float32 and the
    sum is divided by C.
  * epsilon is added to the raw gamma_scale and sigma, which are stored; the
    reconstruction divides out the same float32 sums (gamma_scale+eps) and
    (sigma+eps) that the encoder divided by.
  * Round(Y) rounds half to even.
  * Eq. (4)'s exponent is garbled; the inverse compander is
    l(y) = ((1+alpha)^(y/127) - 1) / alpha, as the notes state and as the
    worked example computes.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

MAG_MAX = 127          # 2^7 - 1, Eq. (3)
NIBBLE_BIAS = 7        # Round-Half-Down bias of Algorithm 1, Stage 4


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def compander(x_abs, alpha):
    """alpha-law compander of the paper's Eq. (3), in float64:
    y = ln(1 + alpha*|x|) / ln(1 + alpha) * (2^7 - 1)."""
    a = np.float64(alpha)
    x = np.asarray(x_abs, dtype=np.float64)
    return np.log1p(a * x) / np.log1p(a) * MAG_MAX


def expander(y, alpha):
    """Inverse compander (paper Eq. (4); notes Eq. (8) and worked example
    Eq. (14)), in float64: |x| = ((1 + alpha)^(y/127) - 1) / alpha."""
    a = np.float64(alpha)
    yy = np.asarray(y, dtype=np.float64)
    return (np.power(1.0 + a, yy / MAG_MAX) - 1.0) / a


@dataclass
class Stages:
    """Every intermediate of Algorithm 1 for a batch of pages [N, H, P]."""
    gmin: np.ndarray      # [N, H]       float32  (Stage 1)
    gscale: np.ndarray    # [N, H]       float32  (Stage 1)
    xn: np.ndarray        # [N, H, P]    float32  (Stage 1)
    mu: np.ndarray        # [N, H, P/C]  float32  (Stage 2)
    xcent: np.ndarray     # [N, H, P/C, C] float32 (Stage 2)
    sigma: np.ndarray     # [N, H, P/C]  float32  (Stage 2)
    xfinal: np.ndarray    # [N, H, P/C, C] float32 (Stage 2)
    Y: np.ndarray         # [N, H, P]    float64  (Stage 3)
    I: np.ndarray         # [N, H, P]    int32    (Stage 3)
    S: np.ndarray         # [N, H, P]    int32 +-1 (Stage 3)


def normalise(x: np.ndarray, C: int, eps, valid=None) -> tuple:
    """Stages 1 and 2 of Algorithm 1 on float32 pages x[N, H, P].

    Stage 1: per channel (row) of a page, gamma_min = min over the
    P tokens, gamma_scale = max - gamma_min, X <- (X - gamma_min) / (gamma_scale + eps).
    Stage 2: view each row as P/C chunks of C tokens; mu = mean of a
    chunk, X_cent = X - mu, sigma = max |X_cent| over the chunk,
    X_final = X_cent / (sigma + eps).

    valid[N] (optional; a partial last page of a sequence): only tokens
    t < valid[n] of page n enter the statistics.  gamma_min / gamma_scale are
    taken over them (0 and 0 for an empty page); a chunk's mu is the
    left-to-right float32 sum of its valid x_n divided by their count, sigma
    the largest |x_n - mu| among them (mu = sigma = 0 for a chunk without
    valid tokens); tokens past valid[n] get X_cent = X_final = 0 (code 0,
    positive sign).  With every valid[n] = P this is the full-page rule.
    """
    x = np.asarray(x, dtype=np.float32)
    N, H, P = x.shape
    assert P % C == 0
    e = np.float32(eps)
    if valid is None:
        gmin = x.min(axis=2)
        gscale = x.max(axis=2) - gmin
        xn = (x - gmin[:, :, None]) / (gscale + e)[:, :, None]
        xv = xn.reshape(N, H, P // C, C)
        s = xv[..., 0].copy()
        for j in range(1, C):                 # left-to-right float32 sum
            s = s + xv[..., j]
        mu = s / np.float32(C)
        xcent = xv - mu[..., None]
        sigma = np.abs(xcent).max(axis=3)
        xfinal = xcent / (sigma + e)[..., None]
        return gmin, gscale, xn, mu, xcent, sigma, xfinal
    v = np.asarray(valid, dtype=np.int64).reshape(N, 1, 1)
    assert np.all((v >= 0) & (v <= P))
    m = np.arange(P)[None, None, :] < v                      # [N, 1, P]
    gmin = np.where(m, x, np.float32(np.inf)).min(axis=2)
    gmax = np.where(m, x, np.float32(-np.inf)).max(axis=2)
    empty = v[:, 0, 0] == 0
    gmin[empty] = 0.0
    gmax[empty] = 0.0
    gscale = gmax - gmin
    xs = np.where(m, x, gmin[:, :, None])                    # padding never enters an operation
    xn = (xs - gmin[:, :, None]) / (gscale + e)[:, :, None]
    xv = xn.reshape(N, H, P // C, C)
    mv = np.broadcast_to(m.reshape(N, 1, P // C, C), xv.shape)
    nc = mv.sum(axis=3)
    s = np.zeros(xv.shape[:3], dtype=np.float32)
    for j in range(C):                                        # left-to-right over the valid tokens
        s = np.where(mv[..., j], s + xv[..., j], s)
    with np.errstate(invalid="ignore", divide="ignore"):
        mu = np.where(nc > 0, s / np.maximum(nc, 1).astype(np.float32), np.float32(0)).astype(np.float32)
    xcent = np.where(mv, xv - mu[..., None], np.float32(0)).astype(np.float32)
    sigma = np.abs(xcent).max(axis=3)
    xfinal = xcent / (sigma + e)[..., None]
    return gmin, gscale, xn, mu, xcent, sigma, xfinal


def quantise(xfinal: np.ndarray, alpha):
    """Stage 3: Y = compander(|X_final|) in float64, I = Round(Y)
    (half to even), S = -1 where X_final < 0 else +1."""
    xf = np.asarray(xfinal, dtype=np.float32)
    Y = compander(np.abs(xf).astype(np.float64), np.float32(alpha))
    I = np.rint(Y).astype(np.int32)
    S = np.where(xf < 0, -1, 1).astype(np.int32)
    return Y, I, S


def split_stream(I: np.ndarray, S: np.ndarray):
    """Stage 4 under reading B; returns (Q_anc, Q_res) as int8 in [-8, 7].

    V_mag   = I >> 4                  anchor magnitude, 0..7
    V_recon = (V_mag << 4) + 7        Round-Half-Down bias at the reconstruction point
    Q_res   = V_recon - I             centred signed correction, -8..7
    Q_anc   = V_mag * S + min(S, 0)   sign-aware two's-complement map
    """
    I = np.asarray(I, dtype=np.int32)
    S = np.asarray(S, dtype=np.int32)
    v_mag = I >> 4
    v_recon = (v_mag << 4) + NIBBLE_BIAS
    q_res = v_recon - I
    q_anc = v_mag * S + np.minimum(S, 0)
    return q_anc.astype(np.int8), q_res.astype(np.int8)


def split_stream_literal(I, S) -> dict:
    """Stage 4 of Algorithm 1 exactly as printed (unpacked integers).  Kept
    for the notes' worked example and to show that the printed anchor needs 18
    levels; the library does not use it."""
    I = np.asarray(I, dtype=np.int32)
    S = np.asarray(S, dtype=np.int32)
    i_bias = I + NIBBLE_BIAS
    v_mag = i_bias >> 4
    v_recon = v_mag << 4
    q_res = v_recon - I
    q_anc = v_mag * S + np.minimum(S, 0)
    return {"I_bias": i_bias, "V_mag": v_mag, "V_recon": v_recon, "Q_res": q_res, "Q_anc": q_anc}


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """Two 4-bit two's-complement codes per byte (paper §5): the low nibble
    holds token 2j, the high nibble token 2j+1.  q[..., P] -> uint8[..., P/2]."""
    n = (np.asarray(q).astype(np.int32) & 0xF).astype(np.uint8)
    return (n[..., 0::2] | (n[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(b: np.ndarray) -> np.ndarray:
    """Inverse of pack_nibbles: uint8[..., P/2] -> int8[..., P] in [-8, 7]."""
    b = np.asarray(b, dtype=np.uint8)
    lo = (b & 0xF).astype(np.int32)
    hi = (b >> 4).astype(np.int32)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.int32)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    out = np.where(out >= 8, out - 16, out)
    return out.astype(np.int8)


def meta_size(H: int, P: int, C: int) -> int:
    """float32 scalars of metadata per page: gamma_min[H], gamma_scale[H],
    mu[P/C][H], sigma[P/C][H] (chunk-major: one chunk's H values are contiguous)."""
    return 2 * H + 2 * H * (P // C)


def pack_meta(gmin, gscale, mu, sigma) -> np.ndarray:
    """mu, sigma given as [N, H, P/C]; stored chunk-major."""
    N, H = gmin.shape
    return np.concatenate([gmin, gscale, mu.transpose(0, 2, 1).reshape(N, -1),
                           sigma.transpose(0, 2, 1).reshape(N, -1)], axis=1).astype(np.float32)


def unpack_meta(meta: np.ndarray, H: int, P: int, C: int):
    """Inverse of pack_meta; returns mu, sigma as [N, H, P/C]."""
    meta = np.asarray(meta, dtype=np.float32).reshape(-1, meta_size(H, P, C))
    nb = P // C
    gmin = meta[:, :H]
    gscale = meta[:, H:2 * H]
    mu = meta[:, 2 * H:2 * H + H * nb].reshape(-1, nb, H).transpose(0, 2, 1)
    sigma = meta[:, 2 * H + H * nb:].reshape(-1, nb, H).transpose(0, 2, 1)
    return gmin, gscale, mu, sigma


def run_stages(x_bits: np.ndarray, alpha, eps, C: int = 32, valid=None) -> Stages:
    """All intermediates of Algorithm 1 for BF16 pages x_bits[N, H, P]
    (valid: optional per-page count of valid tokens, see ``normalise``)."""
    x = bf16_to_f32(x_bits)
    N, H, P = x.shape
    gmin, gscale, xn, mu, xcent, sigma, xfinal = normalise(x, C, eps, valid)
    Y, I, S = quantise(xfinal.reshape(N, H, P), alpha)
    return Stages(gmin, gscale, xn, mu, xcent, sigma, xfinal, Y, I, S)


def encode_pages(x_bits: np.ndarray, alpha, eps, C: int = 32, return_stages: bool = False, valid=None):
    """Algorithm 1 on BF16 pages [N, H, P]; returns (anchor, residual, meta).

    anchor, residual: uint8 [N, H, P/2] packed planes; meta: float32
    [N, 2H + 2H*P/C] = gamma_min[H], gamma_scale[H], mu[P/C][H], sigma[P/C][H].
    valid[N] (optional): per-page count of valid tokens (partial last pages).
    """
    st = run_stages(x_bits, alpha, eps, C, valid)
    q_anc, q_res = split_stream(st.I, st.S)
    anchor = pack_nibbles(q_anc)
    residual = pack_nibbles(q_res)
    meta = pack_meta(st.gmin, st.gscale, st.mu, st.sigma)
    if return_stages:
        return anchor, residual, meta, st
    return anchor, residual, meta


def pages_from_tokens(x_tm_bits: np.ndarray, n_heads: int, H: int = 128, P: int = 256):
    """KV held token-major, as paged attention keeps it, -> the encoder's pages.

    The paper encodes KV pages in a layout that complies with paged attention
    (§4.1, "Hierarchical Quantization"); there the cache is token-major: token
    t's H channels of head h are columns h*H .. h*H + H - 1 of row t.
    x_tm_bits: BF16 bits [n_tokens, >= n_heads * H] (columns past n_heads * H
    are ignored).  Returns (pages [n_heads * n_pp, H, P], valid [n_heads * n_pp])
    with n_pp = ceil(n_tokens / P): page h * n_pp + j holds tokens
    j*P .. j*P + P - 1 of head h channel-major; the last page of each head holds
    the remaining tokens, zero padded, and valid counts them.
    """
    n_tokens = x_tm_bits.shape[0]
    n_pp = -(-n_tokens // P)
    pages = np.zeros((n_heads * n_pp, H, P), dtype=np.uint16)
    valid = np.zeros(n_heads * n_pp, dtype=np.int32)
    for h in range(n_heads):
        for j in range(n_pp):
            t0, t1 = j * P, min((j + 1) * P, n_tokens)
            pages[h * n_pp + j, :, :t1 - t0] = x_tm_bits[t0:t1, h * H:(h + 1) * H].T
            valid[h * n_pp + j] = t1 - t0
    return pages, valid


def encode_tokens(x_tm_bits: np.ndarray, n_heads: int, alpha, eps, C: int = 32):
    """Algorithm 1 on token-major KV: the pages of pages_from_tokens, each last
    page of a head encoded over its valid tokens; returns (anchor, residual, meta)."""
    pages, valid = pages_from_tokens(x_tm_bits, n_heads)
    return encode_pages(pages, alpha, eps, C, valid=valid)


def reconstruct(anchor: np.ndarray, residual, meta: np.ndarray, alpha, eps,
                H: int = 128, P: int = 256, C: int = 32) -> np.ndarray:
    """Inverse transform, float64 result [N, H, P].

    Anchor phase (draft KV; paper §4.2, notes Eq. (14)): from Q_anc alone the
    magnitude index is V_recon = 16*V + 7.  Residual phase (verification KV;
    paper §4.2, notes Eq. (15)): I = V_recon - Q_res.  Then
        x_final = S * l(I)
        x_norm  = x_final * (sigma + eps) + mu
        x       = x_norm * (gamma_scale + eps) + gamma_min
    where (sigma + eps) and (gamma_scale + eps) are the float32 sums the encoder
    divided by.  ``residual=None`` selects the anchor-only reconstruction.
    """
    q_anc = unpack_nibbles(anchor).astype(np.int32)
    N = q_anc.shape[0]
    S = np.where(q_anc < 0, -1, 1)
    v_mag = np.where(S > 0, q_anc, -q_anc - 1)          # inverse of the two's-complement map
    idx = (v_mag << 4) + NIBBLE_BIAS
    if residual is not None:
        idx = idx - unpack_nibbles(residual).astype(np.int32)
    xf = S * expander(idx, np.float32(alpha))
    gmin, gscale, mu, sigma = unpack_meta(meta, H, P, C)
    e = np.float32(eps)
    d_sigma = (sigma + e).astype(np.float64)            # [N, H, P/C]
    d_gamma = (gscale + e).astype(np.float64)           # [N, H]
    xf = xf.reshape(N, H, P // C, C)
    xn = xf * d_sigma[..., None] + mu.astype(np.float64)[..., None]
    x = xn.reshape(N, H, P) * d_gamma[..., None] + gmin.astype(np.float64)[..., None]
    return x
