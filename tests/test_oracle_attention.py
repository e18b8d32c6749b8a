"""Pins of the float64 attention oracle (no GPU).

The oracle is the textbook softmax(q k^T * scale) v; these tests tie it to an
independent implementation (torch's scaled_dot_product_attention in float64
on the CPU), to closed forms, and to the paged / grouped / causal indexing.
"""
import numpy as np
import pytest
import torch

from oracle import attention as at


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(causal):
    R, L, D = 12, 300, 128
    q, k, v = _rand((R, D), 1), _rand((L, D), 2), _rand((L, D), 3)
    scale = D ** -0.5
    nv = (L - R + 1 + np.arange(R)) if causal else None
    o, lse = at.attention_rows(q, k, v, scale, nv)
    mask = None
    if causal:
        mask = torch.from_numpy(np.arange(L)[None, :] < nv[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=None if mask is None else mask[None], scale=scale)[0].numpy()
    assert np.max(np.abs(o - ref)) < 1e-12
    s = torch.from_numpy(q) @ torch.from_numpy(k).T * scale
    if causal:
        s = s.masked_fill(~mask, float("-inf"))
    assert np.max(np.abs(lse - torch.logsumexp(s, dim=1).numpy())) < 1e-12


def test_closed_forms():
    D = 128
    v = _rand((50, D), 4)
    q = _rand((3, D), 5)
    # identical keys: uniform weights, output is the mean of v, lse = s + ln L
    k = np.tile(_rand((1, D), 6), (50, 1))
    o, lse = at.attention_rows(q, k, v, 0.1)
    assert np.max(np.abs(o - v.mean(axis=0))) < 1e-12
    assert np.max(np.abs(lse - (0.1 * q @ k[0] + np.log(50)))) < 1e-12
    # a single visible key returns its value row
    o1, lse1 = at.attention_rows(q, _rand((50, D), 7), v, 0.1, np.array([1, 1, 1]))
    assert np.max(np.abs(o1 - v[0])) < 1e-12


def test_lse_merge_of_two_halves():
    D, L = 128, 512
    q, k, v = _rand((4, D), 8), _rand((L, D), 9), _rand((L, D), 10)
    o, lse = at.attention_rows(q, k, v, 0.09)
    o1, l1 = at.attention_rows(q, k[:200], v[:200], 0.09)
    o2, l2 = at.attention_rows(q, k[200:], v[200:], 0.09)
    m = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - m), np.exp(l2 - m)
    merged = (o1 * w1[:, None] + o2 * w2[:, None]) / (w1 + w2)[:, None]
    assert np.max(np.abs(merged - o)) < 1e-12
    assert np.max(np.abs(m + np.log(w1 + w2) - lse)) < 1e-12


def test_paged_grouped_causal_indexing():
    """V pages carry (kv head, token index) so the output reveals which keys and
    which KV head each query row saw; q = 0 gives uniform weights."""
    B, T, Hkv, G, D = 2, 3, 2, 4, 128
    Hq = Hkv * G
    ctx = np.array([700, 512])
    npages = 3
    table = np.zeros((B, Hkv, npages), dtype=np.int32)
    store = {}
    pid = 0
    for b in range(B):
        for h in range(Hkv):
            for p in range(npages):
                tok = p * 256 + np.arange(256)
                page = np.zeros((D, 256))
                page[0] = tok                 # channel 0: token position
                page[1] = 1000 * h + b        # channel 1: which head / sequence
                store[pid] = page
                table[b, h, p] = pid
                pid += 1
    fetch = lambda ids: (np.stack([store[i] for i in ids]), np.stack([store[i] for i in ids]))
    q = np.zeros((B, T, Hq, D))
    for causal in (False, True):
        o, lse = at.decode_attention(q, fetch, table, ctx, Hkv, 0.1, causal)
        for b in range(B):
            for t in range(T):
                for hq in range(Hq):
                    nvis = ctx[b] - T + t + 1 if causal else ctx[b]
                    assert abs(o[b, t, hq, 0] - (nvis - 1) / 2) < 1e-9
                    assert abs(o[b, t, hq, 1] - (1000 * (hq // G) + b)) < 1e-9
                    assert abs(lse[b, t, hq] - np.log(nvis)) < 1e-9


def test_rows_without_visible_keys():
    q, k, v = _rand((3, 128), 11), _rand((5, 128), 12), _rand((5, 128), 13)
    o, lse = at.attention_rows(q, k, v, 0.1, np.array([0, 2, 5]))
    assert np.all(np.isnan(o[0])) and lse[0] == -np.inf
    o2, l2 = at.attention_rows(q[1:], k[:2], v[:2], 0.1)
    assert np.max(np.abs(o[1] - o2[0])) < 1e-12 and abs(lse[1] - l2[0]) < 1e-12
    oe, le = at.attention_rows(q, k[:0], v[:0], 0.1)
    assert np.all(np.isnan(oe)) and np.all(np.isneginf(le))


def test_vnmse_closed_forms():
    """vNMSE is zero for identical outputs, 1 for o = 2 o_ref and 0.25 for
    o = o_ref / 2 (per-row ||.||^2 ratios), averages rows with equal weight,
    and does not change when every row of both outputs is scaled alike."""
    rng = np.random.default_rng(5)
    r = rng.standard_normal((6, 128))
    assert at.vnmse(r, r) == 0.0
    assert at.vnmse(2 * r, r) == pytest.approx(1.0)
    assert at.vnmse(0.5 * r, r) == pytest.approx(0.25)
    o = r.copy()
    o[0] *= 3.0                                  # one row off by ||2r||^2/||r||^2 = 4
    assert at.vnmse(o, r) == pytest.approx(4.0 / 6)
    s = rng.uniform(0.1, 10.0, (6, 1))
    assert at.vnmse(o * s, r * s) == pytest.approx(at.vnmse(o, r))
    assert at.vnmse(o.reshape(2, 3, 128), r.reshape(2, 3, 128)) == pytest.approx(at.vnmse(o, r))
