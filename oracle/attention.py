"""float64 CPU oracle of decode / verification attention over paged KV.

TEST INFRASTRUCTURE ONLY (imported by the tests, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU legs; never by the library).

The attention is the textbook definition the Lynx paper states in §2.1,
O = softmax(Q K^T / sqrt(d_k)) V (also the reading notes' Eq. (1)), written out
in float64 with a library matmul and exp.  The paper's decode instance runs it
over the dequantised KV pages (§4.2, Anchor phase: draft decode; Residual
phase: one parallel verification pass over the draft tokens, §4.3).

Readings: query heads are grouped onto KV heads in consecutive groups of
G = Hq / Hkv; for T verification tokens with causal masking, query token i
sees keys 0 .. ctx_len - T + i (the drafts occupy the last T positions); the
log-sum-exp returned is the natural log of sum_j exp(scale * q.k_j).
"""
from __future__ import annotations

import numpy as np


def attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                   n_visible: np.ndarray | None = None):
    """softmax(scale * q k^T) v for query rows q[R, D] over keys k[L, D], v[L, D].

    ``n_visible[r]`` (optional) limits row r to keys 0 .. n_visible[r]-1.
    Returns (o[R, D], lse[R]) in float64.
    A row that sees no key has no softmax: its output is NaN (undefined) and
    its log-sum-exp is -inf (the log of an empty sum).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    R, L = q.shape[0], k.shape[0]
    if L == 0:
        return np.full((R, v.shape[1]), np.nan), np.full(R, -np.inf)
    s = (q @ k.T) * float(scale)
    if n_visible is not None:
        cols = np.arange(L)[None, :]
        s = np.where(cols < np.asarray(n_visible)[:, None], s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        o = (p @ v) / l
        lse = (m + np.log(l))[:, 0]
    empty = ~np.isfinite(m[:, 0])
    o[empty] = np.nan
    lse[empty] = -np.inf
    return o, lse


def pages_to_seq(pages: np.ndarray) -> np.ndarray:
    """Channel-major pages [n, 128, 256] -> token-major sequence [n*256, 128]."""
    pages = np.asarray(pages)
    n, H, P = pages.shape
    return pages.transpose(0, 2, 1).reshape(n * P, H)


def decode_attention(q: np.ndarray, kv_pages, page_table: np.ndarray, ctx_len: np.ndarray,
                     n_kv_heads: int, scale: float, causal: bool,
                     batches=None, q_heads=None):
    """Attention of queries q[B, T, Hq, D] over a paged KV cache.

    ``kv_pages(page_ids) -> (k_pages, v_pages)`` returns the dequantised (or
    BF16) K and V pages, float arrays [len(page_ids), D, 256], for the given
    page ids.  ``page_table[b, h, p]`` is the id of logical page p of KV head h
    in sequence b; ``ctx_len[b]`` is the number of valid keys.  ``batches`` and
    ``q_heads`` optionally restrict the computation to a subset (the other
    outputs are left as NaN).  Returns (o[B, T, Hq, D], lse[B, T, Hq]).
    """
    q = np.asarray(q, dtype=np.float64)
    B, T, Hq, D = q.shape
    G = Hq // n_kv_heads
    o = np.full((B, T, Hq, D), np.nan)
    lse = np.full((B, T, Hq), np.nan)
    bs = range(B) if batches is None else batches
    hs = range(Hq) if q_heads is None else q_heads
    for b in bs:
        L = int(ctx_len[b])
        n_pages = -(-L // 256)
        for hk in sorted({hq // G for hq in hs}):
            kp, vp = kv_pages(np.asarray(page_table[b, hk, :n_pages]))
            k = pages_to_seq(kp)[:L]
            v = pages_to_seq(vp)[:L]
            heads = [hq for hq in hs if hq // G == hk]
            rows = q[b][:, heads, :].reshape(T * len(heads), D)
            if causal:
                nv = np.repeat(L - T + 1 + np.arange(T), len(heads))
            else:
                nv = None
            oo, ll = attention_rows(rows, k, v, scale, nv)
            o[b][:, heads, :] = oo.reshape(T, len(heads), D)
            lse[b][:, heads] = ll.reshape(T, len(heads))
    return o, lse


def vnmse(o: np.ndarray, o_ref: np.ndarray) -> float:
    """Compression error of attention outputs as the Lynx paper measures it
    (§6.3 "Compression error", the vNMSE it reports in Table 3): the mean over
    output rows (every query token and head) of ||o - o_ref||^2 / ||o_ref||^2,
    with o the output over compressed KV and o_ref the output over the
    uncompressed KV.  Rows are the last axis; float64."""
    o = np.asarray(o, dtype=np.float64).reshape(-1, np.shape(o)[-1])
    r = np.asarray(o_ref, dtype=np.float64).reshape(-1, np.shape(o_ref)[-1])
    return float(np.mean(np.sum((o - r) ** 2, axis=1) / np.sum(r ** 2, axis=1)))
