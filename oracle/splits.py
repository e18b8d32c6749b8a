"""Plain CPU oracle of the split stream at other Anchor / Residual widths
(3+5, 5+3, 6+2, ...), the alternative bit allocations the Lynx paper leaves to
future work.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  The
library never calls it and shares no code, tables or constants with the CUDA
path.  Every function is pinned (tests/test_oracle_splits.py): the 4+4 split
reproduces the paper's split stream exactly, and the others are checked
against the definition of the 8-bit code and brute-force bit positions.

Sources (cited by page title and section; no code is taken from them):
  [paper] "Lynx: Progressive Speculative Quantization for accelerating KV
          Transfer in Long-Context Inference": §4.1 Algorithm 1 Stage 4 and
          "Split-Stream Construction" (the 4+4 split of the 8-bit code); §8
          (other widths for the two streams, e.g. INT6 or INT2, are possible
          and left to future work).
  [notes] Zhongzhu Zhou's reading notes on the paper: the bit allocations
          3+5, 4+4, 5+3 and 6+2 as the Anchor/Residual splits to explore.

Reading (the pages give only the 4+4 split; listed in the design notes): an
A-bit Anchor (sign included) and an R = 8 - A bit Residual split the 8-bit code
q8 = S > 0 ? I : -I - 1 (I in 0..127) exactly as reading B splits it for A = 4:
  Anchor      Q_anc = q8 >> R (arithmetic), i.e. V = I >> R, Q_anc = S > 0 ? V : -V - 1
  Anchor-only I_hat = V 2^R + 2^(R-1) - 1 (the bin's middle, rounded down; 16V + 7
              for R = 4)
  Residual    Q_res = I_hat - I, in -2^(R-1) .. 2^(R-1) - 1
  Full        I = I_hat - Q_res
Packing: per 32-token chunk, a little-endian bit string of 32 A (resp. 32 R)
bits = 4A (4R) bytes, token t's two's-complement code at bits A t .. A t + A - 1
(the nibble layout of the paper's §5 when A = 4); a channel row of a page holds
its 8 chunks' strings in order (32 A bytes).
"""
from __future__ import annotations

import numpy as np

from oracle import lynx_oracle as lo

MAG_BITS = 7


def split_codes(I: np.ndarray, S: np.ndarray, anchor_bits: int):
    """(Q_anc, Q_res) as int32 for 8-bit codes (I, S) and an A-bit Anchor."""
    A = anchor_bits
    R = 8 - A
    assert 2 <= A <= 7
    V = I >> R
    q_anc = np.where(S > 0, V, -V - 1)
    i_hat = (V << R) + (1 << (R - 1)) - 1
    return q_anc.astype(np.int32), (i_hat - I).astype(np.int32)


def pack_bits(codes: np.ndarray, bits: int, C: int = 32) -> np.ndarray:
    """Signed codes [..., P] (each in -2^(bits-1) .. 2^(bits-1) - 1) -> bytes
    [..., P * bits / 8]: per C-token chunk a little-endian bit string, token t's
    two's-complement code at bits bits * t .. bits * t + bits - 1."""
    c = np.asarray(codes, dtype=np.int64) & ((1 << bits) - 1)
    P = c.shape[-1]
    lead = c.shape[:-1]
    ch = c.reshape(lead + (P // C, C))
    nb = C * bits
    bitarr = ((ch[..., :, None] >> np.arange(bits)) & 1).reshape(lead + (P // C, nb))   # bit i of token t at t*bits+i
    byts = np.zeros(lead + (P // C, nb // 8), dtype=np.uint8)
    for k in range(8):
        byts |= (bitarr[..., k::8] << k).astype(np.uint8)
    return byts.reshape(lead + (P * bits // 8,))


def unpack_bits(b: np.ndarray, bits: int, C: int = 32) -> np.ndarray:
    """Inverse of pack_bits: bytes [..., P * bits / 8] -> int32 [..., P]."""
    b = np.asarray(b, dtype=np.uint8)
    lead = b.shape[:-1]
    nbytes = b.shape[-1]
    P = nbytes * 8 // bits
    ch = b.reshape(lead + (P // C, C * bits // 8))
    bitarr = ((ch[..., :, None] >> np.arange(8)) & 1).reshape(lead + (P // C, C * bits))
    v = (bitarr.reshape(lead + (P // C, C, bits)) << np.arange(bits)).sum(axis=-1)
    v = np.where(v >= 1 << (bits - 1), v - (1 << bits), v)
    return v.reshape(lead + (P,)).astype(np.int32)


def encode_pages_split(x_bits: np.ndarray, anchor_bits: int, alpha, eps, C: int = 32):
    """Algorithm 1 with an A-bit Anchor: (anchor bytes [N, H, P A / 8], residual
    bytes [N, H, P R / 8], meta float32 [N, 2304])."""
    st = lo.run_stages(x_bits, alpha, eps, C)
    qa, qr = split_codes(st.I, st.S, anchor_bits)
    meta = lo.pack_meta(st.gmin, st.gscale, st.mu, st.sigma)
    return pack_bits(qa, anchor_bits, C), pack_bits(qr, 8 - anchor_bits, C), meta


def reconstruct_split(anchor: np.ndarray, residual, meta: np.ndarray, anchor_bits: int, alpha, eps,
                      H: int = 128, P: int = 256, C: int = 32) -> np.ndarray:
    """Anchor-only (residual None) or full reconstruction, float64 [N, H, P]."""
    A = anchor_bits
    R = 8 - A
    qa = unpack_bits(anchor, A, C)
    S = np.where(qa < 0, -1, 1)
    V = np.where(S > 0, qa, -qa - 1)
    idx = (V << R) + (1 << (R - 1)) - 1
    if residual is not None:
        idx = idx - unpack_bits(residual, R, C)
    xf = S * lo.expander(idx, np.float32(alpha))
    N = xf.shape[0]
    gmin, gscale, mu, sigma = lo.unpack_meta(meta, H, P, C)
    e = np.float32(eps)
    xn = xf.reshape(N, H, P // C, C) * (sigma + e).astype(np.float64)[..., None] + mu.astype(np.float64)[..., None]
    return xn.reshape(N, H, P) * (gscale + e).astype(np.float64)[..., None] + gmin.astype(np.float64)[..., None]
