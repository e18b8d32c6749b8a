"""GPU parity of lynx_decode_attn / lynx_decode_attn_bf16 against the float64
attention oracle over the oracle's own dequantised KV.

The page pools fed to the GPU are the oracle's encoding of seeded BF16 pages
(inputs flow oracle -> GPU only), so the comparison isolates the attention
kernel.  Bar: |gpu - oracle| <= 2e-3 * max(1, |oracle|) for outputs and
log-sum-exps.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as at
from oracle import lynx_oracle as lo
from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L

from lynx_testutil import EPS, check_attention, check_codes

pytestmark = pytest.mark.gpu


class Pools:
    """K and V page pools encoded by the oracle, plus their dequantised float64
    copies (anchor-only and full) and the BF16 originals."""

    def __init__(self, n_heads, n_tokens, seed, alpha=100.0, lazy=False):
        out = inputs.outlier_pairs(n_heads, seed)
        self.alpha = alpha
        self.lazy = lazy
        self.kb = inputs.kv_pages_np(n_heads, n_tokens, seed * 10 + 1, out)
        self.vb = inputs.kv_pages_np(n_heads, n_tokens, seed * 10 + 2, out)
        self.n = self.kb.shape[0]
        self.enc = {}
        self.deq = {}
        for name, bits in (("k", self.kb), ("v", self.vb)):
            a, r, m = lo.encode_pages(bits, alpha, EPS)
            self.enc[name] = (a, r, m)
            if lazy:
                continue
            self.deq[(name, "anchor")] = lo.reconstruct(a, None, m, alpha, EPS)
            self.deq[(name, "full")] = lo.reconstruct(a, r, m, alpha, EPS)
            self.deq[(name, "bf16")] = lo.bf16_to_f32(bits).astype(np.float64)
        self.dev = {name: tuple(torch.from_numpy(t).cuda() for t in self.enc[name]) for name in ("k", "v")}
        self.dev_bf16 = {name: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
                         for name, b in (("k", self.kb), ("v", self.vb))}

    def pages(self, name, mode, ids):
        if not self.lazy:
            return self.deq[(name, mode)][ids]
        if mode == "bf16":
            return lo.bf16_to_f32((self.kb if name == "k" else self.vb)[ids]).astype(np.float64)
        a, r, m = self.enc[name]
        return lo.reconstruct(a[ids], r[ids] if mode == "full" else None, m[ids], self.alpha, EPS)

    def fetch(self, mode):
        return lambda ids: (self.pages("k", mode, ids), self.pages("v", mode, ids))


def run(pools, mode, q_bits, table, ctx, Hkv, causal, scale=None):
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    pt = torch.from_numpy(table.astype(np.int32)).cuda()
    cl = torch.from_numpy(ctx.astype(np.int32)).cuda()
    if mode == "bf16":
        o, lse = L.lynx_decode_attn_bf16(q, pools.dev_bf16["k"], pools.dev_bf16["v"], pt, cl, Hkv,
                                         sm_scale=scale, causal=causal)
    else:
        ka, kr, km = pools.dev["k"]
        va, vr, vm = pools.dev["v"]
        full = mode == "full"
        o, lse = L.lynx_decode_attn(q, ka, kr if full else None, km, va, vr if full else None, vm,
                                    pt, cl, Hkv, L.Params(alpha=pools.alpha), sm_scale=scale,
                                    causal=causal)
    torch.cuda.synchronize()
    L.lynx_device_status()
    return o.cpu().numpy(), lse.cpu().numpy()


def reference(pools, mode, q_bits, table, ctx, Hkv, causal, scale=None, **kw):
    q = lo.bf16_to_f32(q_bits).astype(np.float64)
    s = scale if scale is not None else 1.0 / math.sqrt(128)
    return at.decode_attention(q, pools.fetch(mode), table, ctx, Hkv, s, causal, **kw)


def contiguous_table(B, Hkv, pages_per_head, pool_pages_per_head, offset=0):
    t = np.zeros((B, Hkv, pages_per_head), dtype=np.int32)
    for b in range(B):
        for h in range(Hkv):
            t[b, h] = (offset + h * pool_pages_per_head + np.arange(pages_per_head)) % (Hkv * pool_pages_per_head)
    return t


@pytest.fixture(scope="module")
def llama_pools():
    return Pools(8, 16384, 1)


@pytest.mark.parametrize("mode", ["anchor", "full", "bf16"])
def test_llama8b_layer_draft_decode(cuda_device, llama_pools, mode):
    """1-token decode, B=1, 8 KV heads, 32 query heads (GQA 4:1), 16,384 tokens."""
    B, T, Hq, Hkv = 1, 1, 32, 8
    table = contiguous_table(B, Hkv, 64, 64)
    ctx = np.array([16384])
    q = inputs.queries_np((B, T, Hq, 128), 7)
    o, lse = run(llama_pools, mode, q, table, ctx, Hkv, False)
    ro, rl = reference(llama_pools, mode, q, table, ctx, Hkv, False)
    check_attention(o, lse, ro, rl)


@pytest.mark.parametrize("mode", ["anchor", "full", "bf16"])
@pytest.mark.parametrize("T", [4, 8, 32, 33, 48, 64])
def test_verification_causal_ragged_batch(cuda_device, llama_pools, mode, T):
    """T-token causal verification over sequences of different, ragged lengths,
    up to the paper's 64 draft tokens (256 query rows per KV head at G = 4)."""
    B, Hq, Hkv = 3, 32, 8
    ctx = np.array([16384, 5000, 300])
    table = np.stack([contiguous_table(1, Hkv, 64, 64, offset=17 * b)[0] for b in range(B)])
    q = inputs.queries_np((B, T, Hq, 128), 100 + T)
    o, lse = run(llama_pools, mode, q, table, ctx, Hkv, True)
    ro, rl = reference(llama_pools, mode, q, table, ctx, Hkv, True)
    check_attention(o, lse, ro, rl)


@pytest.mark.parametrize("mode", ["anchor", "full", "bf16"])
def test_odd_group_sizes_and_tiny_contexts(cuda_device, llama_pools, mode):
    """G = 3 query heads per KV head (rows not a multiple of 4), T = 3; contexts
    of 1 key, T keys (the first causal row sees a single key) and 0 keys."""
    B, T, Hkv = 4, 3, 2
    Hq = 3 * Hkv
    ctx = np.array([1, 3, 257, 0])
    table = np.stack([contiguous_table(1, Hkv, 2, 64, offset=5 * b)[0] for b in range(B)])
    q = inputs.queries_np((B, T, Hq, 128), 55)
    for causal in (False, True):
        o, lse = run(llama_pools, mode, q, table, ctx, Hkv, causal)
        ro, rl = reference(llama_pools, mode, q, table, np.maximum(ctx, 0), Hkv, causal)
        empty = np.isnan(ro[..., 0])          # rows with no visible key
        assert np.all(o[empty] == 0.0) and np.all(np.isneginf(lse[empty]))
        check_attention(o, lse, np.nan_to_num(ro), rl, mask=~empty)


@pytest.mark.parametrize("mode", ["anchor", "full", "bf16"])
@pytest.mark.parametrize("T", [5, 7])
def test_sixteen_row_tiles_ragged(cuda_device, llama_pools, mode, T):
    """G = 3, T = 5 or 7: 15 or 21 query rows per KV head, so the last 16-row
    tile of the tensor-core path is partly empty and its last 4-row group is
    ragged; contexts include 0 keys, fewer keys than T and a partial page."""
    B, Hkv = 5, 2
    Hq = 3 * Hkv
    ctx = np.array([0, T - 2, 1000, 4099, 1])
    table = np.stack([contiguous_table(1, Hkv, 20, 64, offset=3 * b)[0] for b in range(B)])
    q = inputs.queries_np((B, T, Hq, 128), 300 + T)
    for causal in (False, True):
        o, lse = run(llama_pools, mode, q, table, ctx, Hkv, causal)
        ro, rl = reference(llama_pools, mode, q, table, ctx, Hkv, causal)
        empty = np.isnan(ro[..., 0])
        assert np.all(o[empty] == 0.0) and np.all(np.isneginf(lse[empty]))
        check_attention(o, lse, np.nan_to_num(ro), rl, mask=~empty)


def test_scale_and_shared_pages(cuda_device, llama_pools):
    """Eight sequences whose page tables point at overlapping pages (as eight
    sequences realised over a multi-layer cache), with a non-default scale."""
    B, T, Hq, Hkv = 8, 1, 32, 8
    table = np.stack([contiguous_table(1, Hkv, 32, 64, offset=4 * b)[0] for b in range(B)])
    ctx = np.full(B, 32 * 256)
    q = inputs.queries_np((B, T, Hq, 128), 9)
    o, lse = run(llama_pools, "anchor", q, table, ctx, Hkv, False, scale=0.05)
    ro, rl = reference(llama_pools, "anchor", q, table, ctx, Hkv, False, scale=0.05)
    check_attention(o, lse, ro, rl)


def test_invalid_page_id_and_context_are_reported(cuda_device, llama_pools):
    """Out-of-pool page ids and out-of-range context lengths are not dereferenced:
    the kernel reads page 0 / clamps and sets the device error word."""
    B, T, Hq, Hkv = 1, 1, 32, 8
    table = contiguous_table(B, Hkv, 4, 64)
    table[0, 3, 1] = 10 ** 6
    q = inputs.queries_np((B, T, Hq, 128), 3)
    with pytest.raises(L.LynxError, match="error word = 2"):
        run(llama_pools, "anchor", q, table, np.array([1024]), Hkv, False)
    with pytest.raises(L.LynxError, match="error word = 3"):
        run(llama_pools, "anchor", q, contiguous_table(B, Hkv, 4, 64), np.array([5000]), Hkv, False)
    L.lynx_device_status()     # cleared by the previous read


def test_end_to_end_encode_then_decode(cuda_device):
    """GPU encode followed by GPU decode over the GPU's own planes, against the
    oracle's encode + reconstruct + attention of the same BF16 pages."""
    Hkv, Hq, n_tok = 4, 16, 4096
    out = inputs.outlier_pairs(Hkv, 4)
    kb = inputs.kv_pages_np(Hkv, n_tok, 41, out)
    vb = inputs.kv_pages_np(Hkv, n_tok, 42, out)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
    ka, kr, km = L.lynx_encode_pages(dev(kb))
    va, vr, vm = L.lynx_encode_pages(dev(vb))
    oka, okr, okm, kst = lo.encode_pages(kb, 100.0, EPS, return_stages=True)
    ova, ovr, ovm, vst = lo.encode_pages(vb, 100.0, EPS, return_stages=True)
    check_codes(ka.cpu().numpy(), kr.cpu().numpy(), oka, okr, kst.Y)
    check_codes(va.cpu().numpy(), vr.cpu().numpy(), ova, ovr, vst.Y)
    T = 8
    table = contiguous_table(1, Hkv, 16, 16)
    ctx = np.array([n_tok])
    qb = inputs.queries_np((1, T, Hq, 128), 77)
    q = dev(qb)
    pt = torch.from_numpy(table).cuda()
    cl = torch.from_numpy(ctx.astype(np.int32)).cuda()
    for full in (False, True):
        o, lse = L.lynx_decode_attn(q, ka, kr if full else None, km, va, vr if full else None, vm, pt, cl, Hkv,
                                    causal=True)
        kd = lo.reconstruct(oka, okr if full else None, okm, 100.0, EPS)
        vd = lo.reconstruct(ova, ovr if full else None, ovm, 100.0, EPS)
        ro, rl = at.decode_attention(lo.bf16_to_f32(qb).astype(np.float64), lambda ids: (kd[ids], vd[ids]),
                                     table, ctx, Hkv, 1 / math.sqrt(128), True)
        check_attention(o.cpu().numpy(), lse.cpu().numpy(), ro, rl)


@pytest.mark.slow
def test_qwen235b_layers_full_context_sampled(cuda_device):
    """Qwen3-235B-A22B-shaped layers at the full 131,072-token context (4 KV
    heads, 16 query heads): GPU encode of the layer's K and V, then the three
    decode calls of the benchmark step over the whole context -- the Anchor
    draft (T = 1), the causal T = 8 verification over the full codes (32 rows
    per KV head) and the BF16 decode (T = 1); four query heads (one per KV head)
    are checked against the oracle, which re-encodes the same BF16 pages."""
    w = inputs.QWEN235B_CACHE
    outl = inputs.outlier_pairs(w.n_kv_heads, 0)
    Hkv, Hq = w.n_kv_heads, w.n_q_heads
    for layer in (0, 93):
        k = inputs.kv_pages_torch(Hkv, w.n_tokens, inputs.layer_seed(0, layer, 0), outl, "cuda")
        v = inputs.kv_pages_torch(Hkv, w.n_tokens, inputs.layer_seed(0, layer, 1), outl, "cuda")
        ka, kr, km = L.lynx_encode_pages(k)
        va, vr, vm = L.lynx_encode_pages(v)
        npph = w.pages_per_head
        table = contiguous_table(1, Hkv, npph, npph)
        ctx = np.array([w.n_tokens])
        pt = torch.from_numpy(table).cuda()
        cl = torch.from_numpy(ctx.astype(np.int32)).cuda()
        kbits = k.view(torch.int16).cpu().numpy().view(np.uint16)
        vbits = v.view(torch.int16).cpu().numpy().view(np.uint16)
        heads = [0, 5, 10, 15]
        sel_h = np.zeros(Hq, dtype=bool)
        sel_h[heads] = True
        enc = {}   # the oracle's planes of each KV head's pages (encoded once)

        def pages(ids, mode):
            if mode == "bf16":
                return (lo.bf16_to_f32(kbits[ids]).astype(np.float64), lo.bf16_to_f32(vbits[ids]).astype(np.float64))
            key = int(ids[0])
            if key not in enc:
                enc[key] = (lo.encode_pages(kbits[ids], 100.0, EPS), lo.encode_pages(vbits[ids], 100.0, EPS))
            (oa, orr, om), (ova, ovr, ovm) = enc[key]
            full = mode == "full"
            return (lo.reconstruct(oa, orr if full else None, om, 100.0, EPS),
                    lo.reconstruct(ova, ovr if full else None, ovm, 100.0, EPS))

        for mode, T in (("anchor", 1), ("full", 8), ("bf16", 1)):
            qb = inputs.queries_np((1, T, Hq, 128), 500 + layer + 7 * T)
            q = torch.from_numpy(qb.view(np.int16)).view(torch.bfloat16).cuda()
            causal = T > 1
            if mode == "bf16":
                o, lse = L.lynx_decode_attn_bf16(q, k, v, pt, cl, Hkv, causal=causal)
            else:
                full = mode == "full"
                o, lse = L.lynx_decode_attn(q, ka, kr if full else None, km, va, vr if full else None, vm, pt, cl,
                                            Hkv, causal=causal)
            torch.cuda.synchronize()
            L.lynx_device_status()
            ro, rl = at.decode_attention(lo.bf16_to_f32(qb).astype(np.float64), lambda ids: pages(ids, mode),
                                         table, ctx, Hkv, 1 / math.sqrt(128), causal, q_heads=heads)
            sel = np.zeros(o.shape[:3], dtype=bool)
            sel[:, :, sel_h] = True
            check_attention(o.cpu().numpy(), lse.cpu().numpy(), np.nan_to_num(ro), np.nan_to_num(rl, nan=0.0),
                            mask=sel)
        del k, v, ka, kr, km, va, vr, vm
        torch.cuda.empty_cache()


@pytest.mark.slow
def test_decode_sweep_full_context_sampled(cuda_device):
    """Decode-attention sweep shape: 8 KV heads x 128, 32 query heads, a batch of
    16 sequences whose contexts run from 4,096 to 131,072 tokens (ragged), over
    one pool of oracle-encoded pages; anchor-only at T = 1 and 4, full codes at
    T = 8 and 32 (causal verification), and the BF16 baseline at T = 8.
    Sequences 0, 7 and 15 and query heads 0, 13 and 31 are checked against the
    oracle over the whole context."""
    Hkv, Hq, npph, B = 8, 32, 512, 16
    pools = Pools(Hkv, npph * 256, 7, lazy=True)
    ctx = np.array([4096 + b * 8192 + (37 * b) % 256 for b in range(B)])
    ctx[-1] = npph * 256
    table = np.stack([contiguous_table(1, Hkv, npph, npph, offset=37 * b)[0] for b in range(B)])
    batches, heads = [0, 7, 15], [0, 13, 31]
    for mode, T, causal in (("anchor", 1, False), ("anchor", 4, True), ("full", 8, True),
                            ("full", 32, True), ("bf16", 8, True)):
        q = inputs.queries_np((B, T, Hq, 128), 900 + T)
        o, lse = run(pools, mode, q, table, ctx, Hkv, causal)
        ro, rl = reference(pools, mode, q, table, ctx, Hkv, causal, batches=batches, q_heads=heads)
        sel = np.zeros(o.shape[:3], dtype=bool)
        sel[np.ix_(batches, range(T), heads)] = True
        check_attention(o, lse, np.nan_to_num(ro), np.nan_to_num(rl, nan=0.0), mask=sel)


def test_vnmse_of_anchor_and_full_codes(cuda_device, llama_pools):
    """Compression error of the attention output as the paper measures it
    (vNMSE against the output over the BF16 KV), one-token decode and T = 8
    verification over one Llama-3-8B-shaped layer: the GPU's values agree with
    the oracle's (5% for anchor-only; 30% for full codes, whose error is small
    enough that the kernels' own rounding is a visible part of it) and the full
    codes' error is more than 100x below the anchor-only error."""
    B, Hq, Hkv = 1, 32, 8
    table = contiguous_table(B, Hkv, 64, 64)
    ctx = np.array([16384])
    for T, causal in ((1, False), (8, True)):
        q = inputs.queries_np((B, T, Hq, 128), 21 + T)
        g = {m: run(llama_pools, m, q, table, ctx, Hkv, causal)[0] for m in ("anchor", "full", "bf16")}
        r = {m: reference(llama_pools, m, q, table, ctx, Hkv, causal)[0] for m in ("anchor", "full", "bf16")}
        va_g, va_r = at.vnmse(g["anchor"], g["bf16"]), at.vnmse(r["anchor"], r["bf16"])
        vf_g, vf_r = at.vnmse(g["full"], g["bf16"]), at.vnmse(r["full"], r["bf16"])
        assert va_g == pytest.approx(va_r, rel=0.05)
        assert vf_g == pytest.approx(vf_r, rel=0.3)
        assert vf_r * 100 < va_r and vf_g * 100 < va_g


@pytest.mark.parametrize("mode", ["anchor", "full"])
@pytest.mark.parametrize("T", [9, 12])
def test_thirty_two_row_tiles_ragged(cuda_device, llama_pools, mode, T):
    """G = 4, T = 9 or 12: 36 or 48 query rows per KV head, i.e. one
    full 32-row tensor-core tile (output accumulators in tensor memory) and a
    second one holding 4 or 16 rows; contexts include 0 keys, fewer keys than T
    and partial pages."""
    B, Hkv = 4, 2
    Hq = 4 * Hkv
    ctx = np.array([0, T - 3, 2500, 5121])
    table = np.stack([contiguous_table(1, Hkv, 24, 64, offset=7 * b)[0] for b in range(B)])
    q = inputs.queries_np((B, T, Hq, 128), 400 + T)
    for causal in (False, True):
        o, lse = run(llama_pools, mode, q, table, ctx, Hkv, causal)
        ro, rl = reference(llama_pools, mode, q, table, ctx, Hkv, causal)
        empty = np.isnan(ro[..., 0])
        assert np.all(o[empty] == 0.0) and np.all(np.isneginf(lse[empty]))
        check_attention(o, lse, np.nan_to_num(ro), rl, mask=~empty)


@pytest.mark.parametrize("G,T", [(8, 1), (8, 2), (1, 17), (2, 12)])
def test_bf16_row_tile_boundaries(cuda_device, llama_pools, G, T):
    """BF16 pages: 8 query rows per KV head (one full 8-row tile), 16 (one
    full 16-row tile), 17 (a full 16-row tile and one holding a single row)
    and 24 (a full tile and a half one); causal and not, contexts of 0 keys,
    fewer keys than T, a partial page and several pages."""
    B, Hkv = 4, 2
    Hq = G * Hkv
    ctx = np.array([0, max(T - 3, 1), 2500, 5121])
    table = np.stack([contiguous_table(1, Hkv, 24, 64, offset=5 * b)[0] for b in range(B)])
    q = inputs.queries_np((B, T, Hq, 128), 500 + 10 * G + T)
    for causal in (False, True):
        o, lse = run(llama_pools, "bf16", q, table, ctx, Hkv, causal)
        ro, rl = reference(llama_pools, "bf16", q, table, ctx, Hkv, causal)
        empty = np.isnan(ro[..., 0])
        assert np.all(o[empty] == 0.0) and np.all(np.isneginf(lse[empty]))
        check_attention(o, lse, np.nan_to_num(ro), rl, mask=~empty)


@pytest.mark.parametrize("mode", ["anchor", "full"])
def test_extreme_row_counts_and_alpha(cuda_device, mode):
    """The largest supported row count per KV head (T = 32, G = 8: 256 rows in 8
    32-row tensor-core tiles), plain multi-head attention (G = 1) at T = 1 and eight query heads
    per KV head at T = 1 (one row, and all 8 rows, of a narrow-kernel tile) and
    at T = 12 (the smallest row count the wide tensor-core kernel takes), over
    pools encoded at alpha = 1e4."""
    pools = Pools(2, 2048, 9, alpha=1e4)
    for B, T, Hq, Hkv, causal, ctx in ((1, 32, 16, 2, True, [2048]), (2, 1, 2, 2, False, [1500, 2048]),
                                       (2, 1, 16, 2, False, [2048, 1100]),
                                       (2, 12, 2, 2, True, [700, 2048])):
        table = np.stack([contiguous_table(1, Hkv, 8, 8, offset=b)[0] for b in range(B)])
        ctx = np.array(ctx)
        q = inputs.queries_np((B, T, Hq, 128), 700 + T)
        o, lse = run(pools, mode, q, table, ctx, Hkv, causal)
        ro, rl = reference(pools, mode, q, table, ctx, Hkv, causal)
        check_attention(o, lse, ro, rl)


class ScaledKeys:
    """A pool whose key pages' gamma_min and gamma_scale are multiplied by 2^e
    (keys of magnitude ~2^e; the oracle dequantises the same metadata)."""

    def __init__(self, base, e):
        self.alpha = base.alpha
        self.base = base
        a, r, m = base.enc["k"]
        m = m.copy()
        m[:, :256] *= np.float32(2.0 ** e)
        self.km = m
        self.dev = dict(base.dev)
        self.dev["k"] = (base.dev["k"][0], base.dev["k"][1], torch.from_numpy(m).cuda())

    def fetch(self, mode):
        a, r, _ = self.base.enc["k"]

        def f(ids):
            k = lo.reconstruct(a[ids], r[ids] if mode == "full" else None, self.km[ids], self.alpha, EPS)
            return k, self.base.pages("v", mode, ids)
        return f


@pytest.mark.parametrize("mode,T", [("anchor", 4), ("full", 4), ("full", 8)])
def test_extreme_magnitudes(cuda_device, mode, T):
    """Queries of magnitude 2^24 and 2^-30, keys of magnitude 2^30 and 2^-30
    (the softmax scale compensates, so the logits stay ordinary): the
    tensor-core kernels scale their fp16 operands into range by powers of two
    that return exactly in the softmax scale.  16-row (T = 4) and 32-row
    (T = 8, full codes) tiles."""
    base = Pools(2, 2048, 13, lazy=True)
    B, Hq, Hkv = 2, 8, 2
    ctx = np.array([2048, 1500])
    table = np.stack([contiguous_table(1, Hkv, 8, 8, offset=b)[0] for b in range(B)])
    q0 = lo.bf16_to_f32(inputs.queries_np((B, T, Hq, 128), 950 + T)).astype(np.float64)
    s0 = 1.0 / math.sqrt(128)
    for qe, ke in ((24, 0), (-30, 0), (0, 30), (0, -30)):
        pools = base if ke == 0 else ScaledKeys(base, ke)
        # a BF16 value times a power of two is a BF16 value: keep the top 16 bits
        q_bits = ((q0 * 2.0 ** qe).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        scale = s0 * 2.0 ** (-qe - ke)
        o, lse = run(pools, mode, q_bits, table, ctx, Hkv, True, scale=scale)
        q = lo.bf16_to_f32(q_bits).astype(np.float64)
        ro, rl = at.decode_attention(q, pools.fetch(mode), table, ctx, Hkv, scale, True)
        check_attention(o, lse, ro, rl)


@pytest.mark.parametrize("T", [1, 8])
def test_bf16_extreme_magnitudes(cuda_device, T):
    """BF16 pages with queries of magnitude 2^24 and 2^-30 and keys of 2^30 and
    2^-30 (the softmax scale compensates): BF16 products are exact and sum in
    float32, so only the float32 range matters.  8-row (T = 1) and 16-row
    (T = 8: 32 rows per KV head) tiles."""
    base = Pools(2, 2048, 13, lazy=True)
    B, Hq, Hkv = 2, 8, 2
    ctx = np.array([2048, 1500])
    table = np.stack([contiguous_table(1, Hkv, 8, 8, offset=b)[0] for b in range(B)])
    pt = torch.from_numpy(table.astype(np.int32)).cuda()
    cl = torch.from_numpy(ctx.astype(np.int32)).cuda()
    q0 = lo.bf16_to_f32(inputs.queries_np((B, T, Hq, 128), 960 + T)).astype(np.float64)
    s0 = 1.0 / math.sqrt(128)
    # a BF16 value times a power of two (in range) is a BF16 value: keep the top 16 bits
    scale_bits = lambda x, e: ((x * 2.0 ** e).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    v64 = lo.bf16_to_f32(base.vb).astype(np.float64)
    for qe, ke in ((24, 0), (-30, 0), (0, 30), (0, -30)):
        kbits = scale_bits(lo.bf16_to_f32(base.kb).astype(np.float64), ke)
        qbits = scale_bits(q0, qe)
        scale = s0 * 2.0 ** (-qe - ke)
        q = torch.from_numpy(qbits.view(np.int16)).view(torch.bfloat16).cuda()
        k = torch.from_numpy(kbits.view(np.int16)).view(torch.bfloat16).cuda()
        o, lse = L.lynx_decode_attn_bf16(q, k, base.dev_bf16["v"], pt, cl, Hkv, sm_scale=scale, causal=True)
        torch.cuda.synchronize()
        L.lynx_device_status()
        k64 = lo.bf16_to_f32(kbits).astype(np.float64)
        ro, rl = at.decode_attention(lo.bf16_to_f32(qbits).astype(np.float64), lambda ids: (k64[ids], v64[ids]),
                                     table, ctx, Hkv, scale, True)
        check_attention(o.cpu().numpy(), lse.cpu().numpy(), ro, rl)


@pytest.mark.parametrize("entry", ["anchor", "full_t8", "bf16", "noalloc"])
def test_decode_replays_in_cuda_graph(cuda_device, llama_pools, entry):
    """A decode call captured in a CUDA graph (after one eager call on the
    device) replays to the eager call's results bit for bit: the calls issue
    only kernel launches on the caller's stream.  Draft decode (narrow tiles),
    T = 8 causal verification over full codes (32-row tiles), the BF16 kernel
    and the no-workspace entry point."""
    B, Hq, Hkv = 2, 32, 8
    T = 8 if entry == "full_t8" else 1
    table = torch.from_numpy(np.stack([contiguous_table(1, Hkv, 16, 64, offset=9 * b)[0]
                                       for b in range(B)])).cuda()
    ctx = torch.tensor([4096, 3000], dtype=torch.int32).cuda()
    q = torch.from_numpy(inputs.queries_np((B, T, Hq, 128), 610 + T).view(np.int16)).view(torch.bfloat16).cuda()
    ka, kr, km = llama_pools.dev["k"]
    va, vr, vm = llama_pools.dev["v"]
    ws = torch.empty(max(L.lynx_decode_attn_workspace_size(B, T, Hq, Hkv, 128, 16), 16), dtype=torch.uint8,
                     device="cuda")

    def call(o, lse):
        if entry == "bf16":
            L.lynx_decode_attn_bf16(q, llama_pools.dev_bf16["k"], llama_pools.dev_bf16["v"], table, ctx, Hkv,
                                    out=o, lse=lse, workspace=ws)
        elif entry == "noalloc":
            L.lynx_decode_attn_noalloc(q, ka, None, km, va, None, vm, table, ctx, Hkv, out=o, lse=lse)
        else:
            full = entry == "full_t8"
            L.lynx_decode_attn(q, ka, kr if full else None, km, va, vr if full else None, vm, table, ctx, Hkv,
                               causal=full, out=o, lse=lse, workspace=ws)

    mk = lambda: (torch.empty((B, T, Hq, 128), dtype=torch.float32, device="cuda"),
                  torch.empty((B, T, Hq), dtype=torch.float32, device="cuda"))
    o_e, l_e = mk()
    call(o_e, l_e)
    torch.cuda.synchronize()
    o_g, l_g = mk()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(o_g, l_g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    o_g.zero_()
    l_g.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(o_g, l_g)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    L.lynx_device_status()
    assert torch.equal(o_g, o_e) and torch.equal(l_g, l_e)


def test_back_to_back_calls_share_workspace(cuda_device, llama_pools):
    """Decode calls issued back to back on one stream with one workspace, each
    call's queries written by a kernel right before it: every output equals the
    same call made alone after a device synchronisation.  The decode kernels and
    the split combine are programmatic dependents of the kernel ahead of them;
    this checks that no call reads its inputs or reuses the workspace before the
    kernel ahead has finished."""
    B, Hq, Hkv = 2, 32, 8
    table = torch.from_numpy(np.stack([contiguous_table(1, Hkv, 32, 64, offset=5 * b)[0]
                                       for b in range(B)])).cuda()
    ctx = torch.tensor([8192, 7000], dtype=torch.int32).cuda()
    ka, kr, km = llama_pools.dev["k"]
    va, vr, vm = llama_pools.dev["v"]
    cases = [("anchor", 1), ("full", 8), ("anchor", 4), ("full", 1)]
    qs = [torch.from_numpy(inputs.queries_np((B, T, Hq, 128), 640 + i).view(np.int16)).view(torch.bfloat16).cuda()
          for i, (_, T) in enumerate(cases)]
    n_ws = max(L.lynx_decode_attn_workspace_size(B, T, Hq, Hkv, 128, 32) for _, T in cases)
    ws = torch.empty(max(n_ws, 16), dtype=torch.uint8, device="cuda")

    def call(i, q, o, lse):
        mode, T = cases[i]
        full = mode == "full"
        L.lynx_decode_attn(q, ka, kr if full else None, km, va, vr if full else None, vm, table, ctx, Hkv,
                           causal=T > 1, out=o, lse=lse, workspace=ws)

    outs = [(torch.empty((B, T, Hq, 128), dtype=torch.float32, device="cuda"),
             torch.empty((B, T, Hq), dtype=torch.float32, device="cuda")) for _, T in cases]
    alone = []
    for i in range(len(cases)):
        call(i, qs[i], *outs[i])
        torch.cuda.synchronize()
        alone.append((outs[i][0].clone(), outs[i][1].clone()))
    scratch = [torch.empty_like(q) for q in qs]
    for o, lse in outs:
        o.zero_()
        lse.zero_()
    torch.cuda.synchronize()
    for i in range(len(cases)):
        scratch[i].copy_(qs[i])      # a kernel writes this call's queries just before it
        call(i, scratch[i], *outs[i])
    torch.cuda.synchronize()
    L.lynx_device_status()
    for (o, lse), (oa, la) in zip(outs, alone):
        assert torch.equal(o, oa) and torch.equal(lse, la)


@pytest.mark.parametrize("mode", ["anchor", "full"])
def test_more_than_128_splits(cuda_device, llama_pools, mode):
    """One KV head whose page table lists the pool's 512 key pages twice
    (262,144 keys), 8 query heads, B = 1: the plan takes 147 splits of 7 pages,
    so the split combine gathers more splits than it has threads."""
    ids = np.concatenate([np.arange(512), np.arange(512)]).astype(np.int32)
    table = ids[None, None, :]
    ctx = np.array([262144])
    q = inputs.queries_np((1, 1, 8, 128), 660)
    o, lse = run(llama_pools, mode, q, table, ctx, 1, False)
    ro, rl = reference(llama_pools, mode, q, table, ctx, 1, False)
    check_attention(o, lse, ro, rl)


@pytest.mark.parametrize("mode", ["anchor", "full"])
@pytest.mark.parametrize("T", [1, 2])
def test_rising_scores_across_pages(cuda_device, mode, T):
    """Pages ordered so that each one's largest logit exceeds every earlier
    page's: the running maxima of an online softmax move on nearly every page,
    by leads from below to well above 2^5 depending on the softmax scale (the
    draft kernel moves a maximum only when a score leads it by more than 2^5,
    and otherwise keeps probabilities up to 2^5 times its reference).  Also the
    reverse order, where the maximum is found on the first page and never
    moves."""
    pools = Pools(2, 4096, 21, lazy=True)
    B, Hq, Hkv, npp = 1, 8, 2, 16
    G = Hq // Hkv
    q_bits = inputs.queries_np((B, T, Hq, 128), 960 + T)
    q = lo.bf16_to_f32(q_bits).astype(np.float64)
    ctx = np.array([npp * 256])
    s0 = 1.0 / math.sqrt(128)
    for mult in (1.0, 8.0, 40.0):
        scale = s0 * mult
        for rev in (False, True):
            table = np.zeros((B, Hkv, npp), dtype=np.int32)
            for h in range(Hkv):
                ids = h * npp + np.arange(npp)
                k = pools.pages("k", mode, ids)                  # [npp][128 channels][256 tokens]
                qh = q[0, :, h * G:(h + 1) * G].reshape(-1, 128)  # the rows sharing KV head h
                top = np.einsum("rc,pct->prt", qh, k).max(axis=(1, 2)) * scale
                order = np.argsort(top)
                table[0, h] = ids[order[::-1] if rev else order]
            o, lse = run(pools, mode, q_bits, table, ctx, Hkv, True, scale=scale)
            ro, rl = at.decode_attention(q, pools.fetch(mode), table, ctx, Hkv, scale, True)
            check_attention(o, lse, ro, rl)
