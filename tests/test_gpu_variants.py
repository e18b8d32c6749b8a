"""GPU parity of the single-precision comparators (lynx_encode_variant,
lynx_reconstruct_variant, lynx_decode_attn_int4, lynx_decode_attn_uniform,
lynx_split_nibbles) against oracle/baselines.py, and their consistency with the
split-stream entry points."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as at
from oracle import baselines as bl
from oracle import lynx_oracle as lo
from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L

from lynx_testutil import CODE_EDGE, CODE_FRACTION, EPS, check_attention, check_meta, check_recon, recon_bound

pytestmark = pytest.mark.gpu


def _bf16(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _pages():
    """6 synthetic pages (2 heads x 768 tokens, outlier channels); page 0's first
    rows hold a 16-level ramp and page 1 a constant row."""
    x = inputs.kv_pages_np(2, 768, 61, inputs.outlier_pairs(2, 61))
    x[0, :4] = _bf16((np.arange(256) % 16) * 0.5 - 3.0)
    x[1, 5] = _bf16(np.full(256, 1.75))
    return x


def to_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def check_signed_codes(g, o, Y):
    """Signed codes (S>0 ? I : -I-1): equal except a magnitude step of 1 where the
    oracle's float64 companded value Y is within CODE_EDGE of a rounding edge."""
    g = np.asarray(g, dtype=np.int32)
    o = np.asarray(o, dtype=np.int32)
    diff = g != o
    if diff.any():
        Yd = np.asarray(Y)[diff]
        assert np.all(np.abs(Yd - np.floor(Yd) - 0.5) < CODE_EDGE), "codes differ away from a rounding edge"
        mag = lambda q: np.where(q < 0, -q - 1, q)
        assert np.all(np.abs(mag(g[diff]) - mag(o[diff])) <= 1)
    assert diff.mean() < CODE_FRACTION


def test_lynx_int8_codes_and_reconstruction(cuda_device):
    """Lynx-INT8 codes and metadata against the oracle; on the GPU its bytes
    shifted right by 4 are the Anchor plane of lynx_encode_pages, and its
    reconstruction equals the full-code reconstruction bit for bit."""
    x = _pages()
    xd = to_dev(x)
    codes, meta = L.lynx_encode_variant(xd, "lynx_int8")
    q8 = codes.cpu().numpy().view(np.int8).reshape(-1, 128, 256)
    oq8, ometa = bl.lynx_int8_encode(x, 100.0, EPS)
    st = lo.run_stages(x, 100.0, EPS)
    check_signed_codes(q8, oq8, st.Y)
    check_meta(meta.cpu().numpy(), ometa)
    a, r, m = L.lynx_encode_pages(xd)
    assert torch.equal(m, meta)
    assert np.array_equal(lo.pack_nibbles((q8.astype(np.int32) >> 4).astype(np.int8)), a.cpu().numpy())
    out = L.lynx_reconstruct_variant(codes, meta, "lynx_int8", out_dtype=torch.float32)
    full = L.lynx_reconstruct(a, r, m, out_dtype=torch.float32)
    torch.cuda.synchronize()
    L.lynx_device_status()
    assert torch.equal(out, full)
    check_recon(out.cpu().numpy(), bl.lynx_int8_decode(q8, meta.cpu().numpy(), 100.0, EPS),
                recon_bound(meta.cpu().numpy()), False)


@pytest.mark.parametrize("alpha", [1.0, 100.0, 1e4])
def test_lynx_int4_codes_and_reconstruction(cuda_device, alpha):
    """Lynx-INT4 codes against the oracle's 7-level rounding, metadata equal to
    Algorithm 1's, reconstruction (float32 and BF16) within the float32 bound."""
    x = _pages()
    xd = to_dev(x)
    p = L.Params(alpha=alpha)
    codes, meta = L.lynx_encode_variant(xd, "lynx_int4", p)
    opk, ometa, Y = bl.lynx_int4_encode(x, alpha, EPS, return_y=True)
    g = lo.unpack_nibbles(codes.cpu().numpy().reshape(-1, 128, 128))
    check_signed_codes(g, lo.unpack_nibbles(opk), Y)
    check_meta(meta.cpu().numpy(), ometa)
    _, _, m = L.lynx_encode_pages(xd, p)
    assert torch.equal(m, meta)
    m_np = meta.cpu().numpy()
    ref = bl.lynx_int4_decode(codes.cpu().numpy().reshape(-1, 128, 128), m_np, alpha, EPS)
    for dt, is_bf16 in ((torch.float32, False), (torch.bfloat16, True)):
        out = L.lynx_reconstruct_variant(codes, meta, "lynx_int4", p, out_dtype=dt)
        torch.cuda.synchronize()
        L.lynx_device_status()
        o = out.float().cpu().numpy()
        check_recon(o, ref, recon_bound(m_np), is_bf16)


@pytest.mark.parametrize("bits", [4, 8])
def test_uniform_codes_and_reconstruction(cuda_device, bits):
    """Uniform INT-b: codes and metadata equal to the oracle's (both divide
    correctly rounded and round half to even), reconstruction = fmaf(Q, S, min)
    within one float32 rounding of the float64 value."""
    x = _pages()
    name = f"uniform_int{bits}"
    codes, meta = L.lynx_encode_variant(to_dev(x), name)
    q, mn, sc = bl.uniform_encode(x, bits)
    g = codes.cpu().numpy().reshape(-1, 128, 256 if bits == 8 else 128)
    if bits == 4:
        g = bl.unpack_codes4(g)
    assert np.array_equal(g, q)
    mg = meta.cpu().numpy().reshape(-1, 2, 128)
    assert np.array_equal(mg[:, 0], mn) and np.array_equal(mg[:, 1], sc)
    out = L.lynx_reconstruct_variant(codes, meta, name, out_dtype=torch.float32)
    torch.cuda.synchronize()
    L.lynx_device_status()
    ref = bl.uniform_decode(q, mn, sc)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= 2.0 ** -24 * np.abs(ref) + 1e-30)


def _table(B, Hkv, npph):
    return np.stack([np.stack([(h * npph + np.arange(npph) + b) % (Hkv * npph) for h in range(Hkv)])
                     for b in range(B)]).astype(np.int32)


@pytest.mark.parametrize("T", [1, 8])
def test_lynx_int4_decode_attention(cuda_device, T):
    """Attention over Lynx-INT4 K and V pools (2 KV heads x 2048 tokens, 8
    query heads) encoded by the oracle, through the draft kernels (T = 1: 8-row
    narrow tiles; T = 8 causal: 16-row tensor-core tiles), against the float64
    oracle over the oracle's dequantisation of the same codes."""
    Hkv, Hq, n_tok = 2, 8, 2048
    outl = inputs.outlier_pairs(Hkv, 71)
    pools = {}
    for name, seed in (("k", 711), ("v", 712)):
        bits = inputs.kv_pages_np(Hkv, n_tok, seed, outl)
        opk, ometa = bl.lynx_int4_encode(bits, 100.0, EPS)
        pools[name] = (torch.from_numpy(opk).cuda(), torch.from_numpy(ometa).cuda(),
                       bl.lynx_int4_decode(opk, ometa, 100.0, EPS))
    npph = n_tok // 256
    B = 2
    table = _table(B, Hkv, npph)
    ctx = np.array([2048, 1300], dtype=np.int32)
    q_bits = inputs.queries_np((B, T, Hq, 128), 720 + T)
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    o, lse = L.lynx_decode_attn_int4(q, pools["k"][0], pools["k"][1], pools["v"][0], pools["v"][1],
                                     torch.from_numpy(table).cuda(), torch.from_numpy(ctx).cuda(), Hkv,
                                     causal=T > 1)
    torch.cuda.synchronize()
    L.lynx_device_status()
    fetch = lambda ids: (pools["k"][2][ids], pools["v"][2][ids])
    ro, rl = at.decode_attention(lo.bf16_to_f32(q_bits).astype(np.float64), fetch, table, ctx, Hkv,
                                 1.0 / math.sqrt(128), T > 1)
    check_attention(o.cpu().numpy(), lse.cpu().numpy(), ro, rl)


def test_split_nibbles_matches_the_byte_plane(cuda_device):
    """lynx_split_nibbles on random byte planes: the low- and high-nibble planes
    hold the bytes' nibbles, token 2j in the low half of byte j."""
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, (3, 128, 256), dtype=np.uint8)
    lo_d, hi_d = L.lynx_split_nibbles(torch.from_numpy(codes).cuda())
    torch.cuda.synchronize()
    exp_lo = (codes[..., 0::2] & 15) | ((codes[..., 1::2] & 15) << 4)
    exp_hi = (codes[..., 0::2] >> 4) | ((codes[..., 1::2] >> 4) << 4)
    assert np.array_equal(lo_d.cpu().numpy(), exp_lo) and np.array_equal(hi_d.cpu().numpy(), exp_hi)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("T", [1, 8])
def test_uniform_decode_attention(cuda_device, bits, T):
    """Attention over uniform INT-b K and V pools encoded by the oracle (2 KV
    heads x 2048 tokens, 8 query heads; INT8 codes split into nibble planes on
    the GPU): the draft kernels (T = 1) and the tensor-core tiles (T = 8,
    causal) against the float64 oracle over min + Q * scale."""
    Hkv, Hq, n_tok = 2, 8, 2048
    outl = inputs.outlier_pairs(Hkv, 81)
    pools = {}
    for name, seed in (("k", 811), ("v", 812)):
        xb = inputs.kv_pages_np(Hkv, n_tok, seed + bits, outl)
        qc, mn, sc = bl.uniform_encode(xb, bits)
        meta = torch.from_numpy(np.stack([mn, sc], axis=1).reshape(-1, 256).astype(np.float32)).cuda()
        if bits == 4:
            lo_p, hi_p = torch.from_numpy(bl.pack_codes4(qc)).cuda(), None
        else:
            lo_p, hi_p = L.lynx_split_nibbles(torch.from_numpy(qc).cuda())
        pools[name] = (lo_p, hi_p, meta, bl.uniform_decode(qc, mn, sc))
    npph = n_tok // 256
    B = 2
    table = _table(B, Hkv, npph)
    ctx = np.array([2048, 1500], dtype=np.int32)
    q_bits = inputs.queries_np((B, T, Hq, 128), 830 + T + bits)
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    k, v = pools["k"], pools["v"]
    o, lse = L.lynx_decode_attn_uniform(q, bits, k[0], k[1], k[2], v[0], v[1], v[2],
                                        torch.from_numpy(table).cuda(), torch.from_numpy(ctx).cuda(), Hkv,
                                        causal=T > 1)
    torch.cuda.synchronize()
    L.lynx_device_status()
    fetch = lambda ids: (k[3][ids], v[3][ids])
    ro, rl = at.decode_attention(lo.bf16_to_f32(q_bits).astype(np.float64), fetch, table, ctx, Hkv,
                                 1.0 / math.sqrt(128), T > 1)
    check_attention(o.cpu().numpy(), lse.cpu().numpy(), ro, rl)
