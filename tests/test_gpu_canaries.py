"""Guard bands around every output and workspace buffer of every entry point.

Each buffer a call writes is a view into a larger device allocation whose
first and last 4 KiB hold a fixed byte pattern; after the call (and after the
device has finished) the pattern must be intact.  A store past either end of
a buffer -- anchor, residual, metadata, reconstruction, attention output,
log-sum-exp, split workspace -- shows up here even where the parity tests,
which read only the in-bounds elements, would not see it.  The shapes cover
ragged ends: a partial last 4-row group of query rows, contexts that end
inside a page, and page counts that are not a multiple of a CTA's work.
"""
import numpy as np
import pytest
import torch

from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L

pytestmark = pytest.mark.gpu

GUARD = 4096


class Guarded:
    """Device buffers with guard bands; ``new`` hands out the in-bounds views."""

    def __init__(self):
        self.bufs = []

    def new(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        buf = torch.empty(GUARD + n + GUARD, dtype=torch.uint8, device="cuda")
        pat = (torch.arange(buf.numel(), device="cuda", dtype=torch.int64) * 151 + 89) % 251
        buf.copy_(pat.to(torch.uint8))
        self.bufs.append((buf, pat.to(torch.uint8), n))
        view = buf[GUARD:GUARD + n].view(dtype).view(shape)
        view.zero_()
        return view

    def workspace(self, B, T, Hq, Hkv, max_pages):
        return self.new((max(L.lynx_decode_attn_workspace_size(B, T, Hq, Hkv, 128, max_pages), 16),), torch.uint8)

    def check(self):
        torch.cuda.synchronize()
        L.lynx_device_status()
        for k, (buf, pat, n) in enumerate(self.bufs):
            assert torch.equal(buf[:GUARD], pat[:GUARD]), f"buffer {k}: store before its start"
            assert torch.equal(buf[GUARD + n:], pat[GUARD + n:]), f"buffer {k}: store past its end"


@pytest.fixture(scope="module")
def data(cuda_device):
    Hkv, npph = 2, 5                              # 5 pages per head: splits end on odd page counts
    out = inputs.outlier_pairs(Hkv, 60)
    k = inputs.kv_pages_torch(Hkv, 256 * npph, 61, out, "cuda")
    v = inputs.kv_pages_torch(Hkv, 256 * npph, 62, out, "cuda")
    ka, kr, km = L.lynx_encode_pages(k)
    va, vr, vm = L.lynx_encode_pages(v)
    table = torch.arange(Hkv * npph, dtype=torch.int32, device="cuda").view(1, Hkv, npph).repeat(3, 1, 1)
    ctx = torch.tensor([256 * npph, 1000, 37], dtype=torch.int32, device="cuda")
    return dict(Hkv=Hkv, npph=npph, k=k, v=v, K=(ka, kr, km), V=(va, vr, vm), table=table, ctx=ctx)


def test_encoders_and_reconstructions(data):
    g = Guarded()
    x = data["k"]
    n = x.shape[0]
    L.lynx_encode_pages(x, anchor=g.new((n, 128, 128), torch.uint8), residual=g.new((n, 128, 128), torch.uint8),
                        meta=g.new((n, L.META_FLOATS), torch.float32))
    valid = torch.tensor([256, 255, 1, 0, 129, 33, 256, 2, 200, 31], dtype=torch.int32, device="cuda")[:n]
    L.lynx_encode_pages(x, anchor=g.new((n, 128, 128), torch.uint8), residual=g.new((n, 128, 128), torch.uint8),
                        meta=g.new((n, L.META_FLOATS), torch.float32), valid_tokens=valid)
    n_heads, n_tok = 3, 600                        # token-major input, each head's last page partial
    xt = torch.randn((n_tok, n_heads * 128), device="cuda").to(torch.bfloat16)
    npg = n_heads * ((n_tok + 255) // 256)
    L.lynx_encode_tokens(xt, n_heads, anchor=g.new((npg, 128, 128), torch.uint8),
                         residual=g.new((npg, 128, 128), torch.uint8), meta=g.new((npg, L.META_FLOATS), torch.float32))
    ka, kr, km = data["K"]
    for res in (None, kr):
        for dt in (torch.bfloat16, torch.float32):
            L.lynx_reconstruct(ka, res, km, out=g.new((n, 128, 256), dt), out_dtype=dt)
    mags = torch.rand(1000, device="cuda")
    L.lynx_quantize_magnitudes(mags, codes=g.new((1000,), torch.uint8))
    g.check()


def test_variants_splits_and_nibble_planes(data):
    g = Guarded()
    x = data["k"]
    n = x.shape[0]
    for name, (_, cb, mf) in L.VARIANTS.items():
        codes = g.new((n, cb), torch.uint8)
        meta = g.new((n, mf), torch.float32)
        L.lynx_encode_variant(x, name, codes=codes, meta=meta)
        for dt in (torch.bfloat16, torch.float32):
            L.lynx_reconstruct_variant(codes, meta, name, out=g.new((n, 128, 256), dt), out_dtype=dt)
        if name == "uniform_int8":
            L.lynx_split_nibbles(codes.view(n, 128, 256), lo=g.new((n, 128, 128), torch.uint8),
                                 hi=g.new((n, 128, 128), torch.uint8))
    for A in (2, 3, 5, 6):
        an = g.new((n, 128, 32 * A), torch.uint8)
        rs = g.new((n, 128, 32 * (8 - A)), torch.uint8)
        mt = g.new((n, L.META_FLOATS), torch.float32)
        L.lynx_encode_split(x, A, anchor=an, residual=rs, meta=mt)
        for res in (None, rs):
            L.lynx_reconstruct_split(an, res, mt, A, out=g.new((n, 128, 256), torch.float32),
                                     out_dtype=torch.float32)
    g.check()


@pytest.mark.parametrize("mode,T,G", [("anchor", 1, 4), ("anchor", 1, 3), ("full", 1, 4), ("anchor", 4, 4),
                                      ("full", 8, 4), ("full", 64, 4), ("anchor", 33, 3), ("bf16", 1, 4),
                                      ("bf16", 8, 3)])
def test_decode_outputs_and_workspace(data, mode, T, G):
    """Draft, narrow and verification kernels (8-, 16- and 32-row tiles, up to
    T = 64), and the BF16 kernel; every call's out, lse and workspace guarded."""
    g = Guarded()
    Hkv, B = data["Hkv"], 3
    Hq = G * Hkv
    q = inputs.queries_torch((B, T, Hq, 128), 63 + T, "cuda")
    out, lse = g.new((B, T, Hq, 128), torch.float32), g.new((B, T, Hq), torch.float32)
    ws = g.workspace(B, T, Hq, Hkv, data["npph"])
    ka, kr, km = data["K"]
    va, vr, vm = data["V"]
    for causal in (False, True):
        if mode == "bf16":
            L.lynx_decode_attn_bf16(q, data["k"], data["v"], data["table"], data["ctx"], Hkv, causal=causal,
                                    out=out, lse=lse, workspace=ws)
        else:
            full = mode == "full"
            L.lynx_decode_attn(q, ka, kr if full else None, km, va, vr if full else None, vm, data["table"],
                               data["ctx"], Hkv, causal=causal, out=out, lse=lse, workspace=ws)
    g.check()


def test_comparator_decodes_merge_and_noalloc(data):
    g = Guarded()
    Hkv, B, T = data["Hkv"], 3, 1
    Hq = 4 * Hkv
    q = inputs.queries_torch((B, T, Hq, 128), 64, "cuda")
    n = data["k"].shape[0]
    c4, m4 = L.lynx_encode_variant(data["k"], "lynx_int4")
    d4, n4 = L.lynx_encode_variant(data["v"], "lynx_int4")
    L.lynx_decode_attn_int4(q, c4, m4, d4, n4, data["table"], data["ctx"], Hkv,
                            out=g.new((B, T, Hq, 128), torch.float32), lse=g.new((B, T, Hq), torch.float32),
                            workspace=g.workspace(B, T, Hq, Hkv, data["npph"]))
    for bits in (4, 8):
        name = "uniform_int4" if bits == 4 else "uniform_int8"
        ck, mk = L.lynx_encode_variant(data["k"], name)
        cv, mv = L.lynx_encode_variant(data["v"], name)
        if bits == 8:
            klo, khi = L.lynx_split_nibbles(ck.view(n, 128, 256))
            vlo, vhi = L.lynx_split_nibbles(cv.view(n, 128, 256))
        else:
            klo, khi, vlo, vhi = ck.view(n, 128, 128), None, cv.view(n, 128, 128), None
        L.lynx_decode_attn_uniform(q, bits, klo, khi, mk, vlo, vhi, mv, data["table"], data["ctx"], Hkv,
                                   out=g.new((B, T, Hq, 128), torch.float32), lse=g.new((B, T, Hq), torch.float32),
                                   workspace=g.workspace(B, T, Hq, Hkv, data["npph"]))
    ka, kr, km = data["K"]
    va, vr, vm = data["V"]
    oa, la = L.lynx_decode_attn(q, ka, None, km, va, None, vm, data["table"], data["ctx"], Hkv)
    ob, lb = L.lynx_decode_attn_bf16(q, data["k"], data["v"], data["table"], data["ctx"], Hkv)
    L.lynx_attn_merge(oa, la, ob, lb, out=g.new(oa.shape, torch.float32), lse=g.new(la.shape, torch.float32))
    L.lynx_decode_attn_noalloc(q, ka, None, km, va, None, vm, data["table"], data["ctx"], Hkv,
                               out=g.new((B, T, Hq, 128), torch.float32), lse=g.new((B, T, Hq), torch.float32))
    g.check()
