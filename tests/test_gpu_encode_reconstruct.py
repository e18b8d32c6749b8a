"""GPU parity of lynx_encode_pages and lynx_reconstruct against the CPU oracle.

Inputs are seeded BF16 pages; the oracle encodes the same bits on the CPU.
Codes: bit-exact except +-1 within 1e-5 of a rounding edge (fraction < 1e-4).
Metadata: within 1e-6 relative.  Reconstruction (fed with the oracle's own
planes): within the float32 error bound of the float64 value, plus half a BF16
ulp for BF16 output.
"""
import numpy as np
import pytest
import torch

from oracle import lynx_oracle as lo
from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L

from lynx_testutil import EPS, check_codes, check_meta, check_recon, recon_bound

pytestmark = pytest.mark.gpu


def to_dev(bits: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def encode_and_compare(bits, alpha=100.0):
    x = to_dev(bits)
    a, r, m = L.lynx_encode_pages(x, L.Params(alpha=alpha))
    torch.cuda.synchronize()
    L.lynx_device_status()
    oa, orr, om, st = lo.encode_pages(bits, alpha, EPS, return_stages=True)
    frac = check_codes(a.cpu().numpy(), r.cpu().numpy(), oa, orr, st.Y)
    exact = check_meta(m.cpu().numpy(), om)
    return frac, exact


@pytest.mark.parametrize("alpha", [100.0, 255.0])
def test_single_page(cuda_device, alpha):
    bits = inputs.kv_pages_np(1, 256, 0, inputs.outlier_pairs(1, 0, count=4))
    frac, exact = encode_and_compare(bits, alpha)
    assert exact == 1.0          # same IEEE float32 steps on both sides


def test_llama8b_layer_k_and_v(cuda_device):
    out = inputs.outlier_pairs(8, 0)
    k = inputs.kv_pages_np(8, 16384, 1, out)
    v = inputs.kv_pages_np(8, 16384, 2, out)
    bits = np.concatenate([k, v])
    assert bits.shape == (1024, 128, 256)
    frac, exact = encode_and_compare(bits)
    assert exact == 1.0


@pytest.mark.parametrize("n_pages", [1, 3, 37, 301])
def test_ragged_page_counts(cuda_device, n_pages):
    bits = inputs.kv_pages_np(1, 256 * n_pages, 5 + n_pages, inputs.outlier_pairs(1, 5, count=2))
    encode_and_compare(bits)


def special_pages():
    rng = np.random.default_rng(11)
    pages = []
    x = rng.standard_normal((128, 256)).astype(np.float32)
    x[3] = 1.5                                           # constant channel
    x[4] = np.where(np.arange(256) % 2 == 0, -2.0, 6.0)  # two-level channel
    x[5] = np.arange(256)                                # ramp
    x[6] = 0.0                                           # all zeros
    x[7] = -0.0                                          # negative zeros
    x[8, ::3] = -0.0                                     # mixed signed zeros
    x[9] = rng.standard_normal(256) * 1e-30              # tiny values
    x[10] = rng.standard_normal(256) * 3e4               # large values
    x[11] = 1e-3 * np.round(rng.standard_normal(256) * 4)  # heavy ties
    pages.append(x)
    pages.append(np.full((128, 256), 7.25, dtype=np.float32))             # constant page
    y = rng.laplace(0, 0.1, (128, 256)).astype(np.float32)
    y[:, 100] = 50.0                                                       # single spike per row
    pages.append(y)
    return inputs.f32_to_bf16_bits(np.stack(pages))


@pytest.mark.parametrize("alpha", [0.25, 100.0, 255.0, 1e4])
def test_special_pages(cuda_device, alpha):
    encode_and_compare(special_pages(), alpha)


def test_zero_pages_is_a_noop(cuda_device):
    x = torch.empty((0, 128, 256), dtype=torch.bfloat16, device="cuda")
    a, r, m = L.lynx_encode_pages(x)
    assert a.numel() == 0 and m.numel() == 0


@pytest.mark.slow
def test_qwen32b_cache_full_size_sampled(cuda_device):
    """The 64-layer Qwen-32B-shaped cache (65,536 pages, 4.29e9 BF16 bytes) in one
    launch, as the benchmark runs it; 256 seeded pages are checked against the oracle."""
    w = inputs.QWEN32B_CACHE
    outl = inputs.outlier_pairs(w.n_kv_heads, 0)
    per = w.pages_per_tensor_layer
    x = torch.empty((2 * w.n_layers * per, 128, 256), dtype=torch.bfloat16, device="cuda")
    for layer in range(w.n_layers):
        for t in range(2):
            i = (2 * layer + t) * per
            x[i:i + per] = inputs.kv_pages_torch(w.n_kv_heads, w.n_tokens, inputs.layer_seed(0, layer, t),
                                                 outl, "cuda")
    a, r, m = L.lynx_encode_pages(x)
    torch.cuda.synchronize()
    L.lynx_device_status()
    idx = np.sort(np.random.default_rng(3).choice(x.shape[0], 256, replace=False))
    ti = torch.from_numpy(idx).cuda()
    bits = x[ti].view(torch.int16).cpu().numpy().view(np.uint16)
    oa, orr, om, st = lo.encode_pages(bits, 100.0, EPS, return_stages=True)
    check_codes(a[ti].cpu().numpy(), r[ti].cpu().numpy(), oa, orr, st.Y)
    check_meta(m[ti].cpu().numpy(), om)


# ------------------------------------------------------------------ reconstruct

def oracle_planes(bits, alpha=100.0):
    oa, orr, om = lo.encode_pages(bits, alpha, EPS)
    return oa, orr, om


@pytest.mark.parametrize("full", [False, True])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n_pages,alpha", [(1, 100.0), (37, 255.0), (512, 100.0)])
def test_reconstruct_parity(cuda_device, full, out_dtype, n_pages, alpha):
    bits = inputs.kv_pages_np(1, 256 * n_pages, 21, inputs.outlier_pairs(1, 21, count=3))
    oa, orr, om = oracle_planes(bits, alpha)
    out = L.lynx_reconstruct(torch.from_numpy(oa).cuda(), torch.from_numpy(orr).cuda() if full else None,
                             torch.from_numpy(om).cuda(), L.Params(alpha=alpha), out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = lo.reconstruct(oa, orr if full else None, om, alpha, EPS)
    check_recon(out.float().cpu().numpy(), ref, recon_bound(om), out_dtype == torch.bfloat16)


def test_reconstruct_special_pages(cuda_device):
    bits = special_pages()
    oa, orr, om = oracle_planes(bits)
    for full in (False, True):
        out = L.lynx_reconstruct(torch.from_numpy(oa).cuda(), torch.from_numpy(orr).cuda() if full else None,
                                 torch.from_numpy(om).cuda(), out_dtype=torch.float32)
        ref = lo.reconstruct(oa, orr if full else None, om, 100.0, EPS)
        check_recon(out.cpu().numpy(), ref, recon_bound(om), False)


def test_encode_then_reconstruct_round_trip(cuda_device):
    """The hot path end to end on the GPU: encode, then both reconstructions,
    against the oracle's encode + reconstruct of the same BF16 bits."""
    bits = inputs.kv_pages_np(2, 256 * 16, 31, inputs.outlier_pairs(2, 31, count=3))
    x = to_dev(bits)
    a, r, m = L.lynx_encode_pages(x)
    oa, orr, om, st = lo.encode_pages(bits, 100.0, EPS, return_stages=True)
    check_codes(a.cpu().numpy(), r.cpu().numpy(), oa, orr, st.Y)
    for full in (False, True):
        out = L.lynx_reconstruct(a, r if full else None, m, out_dtype=torch.float32)
        ref = lo.reconstruct(oa, orr if full else None, om, 100.0, EPS)
        # a code that differs by one at a rounding edge moves that element by one code step
        err = np.abs(out.cpu().numpy() - ref) <= recon_bound(om)
        assert err.mean() > 1 - 1e-4


# ---------------------------------------------------------------- partial pages
def test_partial_pages_parity_and_padding_independence(cuda_device):
    """lynx_encode_pages_partial against the oracle's partial-page rule for valid
    counts at and around every chunk edge (0, 1, 31, 32, 33, 77, 128, 255, 256),
    over random padding; pages with 256 valid tokens are byte-identical to
    lynx_encode_pages, and changing the padding changes nothing."""
    counts = np.array([0, 1, 31, 32, 33, 77, 128, 255, 256, 256, 160, 2])
    n = len(counts)
    bits = inputs.kv_pages_np(2, 256 * n // 2, 81, inputs.outlier_pairs(2, 81))
    rng = np.random.default_rng(82)
    for p, v in enumerate(counts):
        bits[p, :, v:] = rng.integers(0, 1 << 16, bits[p, :, v:].shape, dtype=np.uint16) & 0x7F7F
    valid = torch.from_numpy(counts.astype(np.int32)).cuda()
    a, r, m = L.lynx_encode_pages(to_dev(bits), valid_tokens=valid)
    torch.cuda.synchronize()
    L.lynx_device_status()
    oa, orr, om, st = lo.encode_pages(bits, 100.0, EPS, return_stages=True, valid=counts)
    check_codes(a.cpu().numpy(), r.cpu().numpy(), oa, orr, st.Y)
    check_meta(m.cpu().numpy(), om)
    # full pages: the partial kernel reproduces the full-page kernel byte for byte
    fa, fr, fm = L.lynx_encode_pages(to_dev(bits))
    full = np.nonzero(counts == 256)[0]
    assert np.array_equal(a.cpu().numpy()[full], fa.cpu().numpy()[full])
    assert np.array_equal(r.cpu().numpy()[full], fr.cpu().numpy()[full])
    assert np.array_equal(m.cpu().numpy()[full], fm.cpu().numpy()[full])
    # other padding (huge values and non-finite bits): same output
    b2 = bits.copy()
    for p, v in enumerate(counts):
        b2[p, :, v:] = np.where(rng.random(b2[p, :, v:].shape) < 0.5, 0x7F00, 0xFF80)
    a2, r2, m2 = L.lynx_encode_pages(to_dev(b2), valid_tokens=valid)
    assert np.array_equal(a2.cpu().numpy(), a.cpu().numpy())
    assert np.array_equal(r2.cpu().numpy(), r.cpu().numpy())
    assert np.array_equal(m2.cpu().numpy(), m.cpu().numpy())


def test_partial_last_page_then_decode(cuda_device):
    """A 1,000-token sequence (last page 232 tokens) encoded on the GPU with its
    valid counts, then decoded over its anchor and full codes: against the oracle
    over the oracle's encoding of the same pages."""
    from oracle import attention as at
    import math
    Hkv, Hq, ctx = 2, 8, 1000
    out = inputs.outlier_pairs(Hkv, 83)
    kb = inputs.kv_pages_np(Hkv, 1024, 84, out)
    vb = inputs.kv_pages_np(Hkv, 1024, 85, out)
    counts = np.tile(np.array([256, 256, 256, ctx - 768], dtype=np.int32), Hkv)
    valid = torch.from_numpy(counts).cuda()
    ka, kr, km = L.lynx_encode_pages(to_dev(kb), valid_tokens=valid)
    va, vr, vm = L.lynx_encode_pages(to_dev(vb), valid_tokens=valid)
    oka, okr, okm = lo.encode_pages(kb, 100.0, EPS, valid=counts)
    ova, ovr, ovm = lo.encode_pages(vb, 100.0, EPS, valid=counts)
    table = torch.from_numpy(np.array([[[4 * h + p for p in range(4)] for h in range(Hkv)]], dtype=np.int32)).cuda()
    q = inputs.queries_np((1, 1, Hq, 128), 86)
    qd = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda()
    cl = torch.from_numpy(np.array([ctx], dtype=np.int32)).cuda()
    for full in (False, True):
        o, lse = L.lynx_decode_attn(qd, ka, kr if full else None, km, va, vr if full else None, vm, table, cl, Hkv)
        kd = lo.reconstruct(oka, okr if full else None, okm, 100.0, EPS)
        vd = lo.reconstruct(ova, ovr if full else None, ovm, 100.0, EPS)
        ro, rl = at.decode_attention(lo.bf16_to_f32(q).astype(np.float64), lambda ids: (kd[ids], vd[ids]),
                                     table.cpu().numpy(), np.array([ctx]), Hkv, 1 / math.sqrt(128), False)
        from lynx_testutil import check_attention
        check_attention(o.cpu().numpy(), lse.cpu().numpy(), ro, rl)


def test_anchor_stream_as_one_contiguous_block(cuda_device):
    """The Anchor stream as the paper serialises it -- the Anchor planes of all
    pages followed immediately by their metadata, one buffer -- written by
    lynx_encode_pages through two views of that buffer, and read back by the
    reconstruction and the draft decode: results equal those of separate
    buffers."""
    n_heads, n_tok = 2, 2048
    outl = inputs.outlier_pairs(n_heads, 41)
    x = torch.cat([inputs.kv_pages_torch(n_heads, n_tok, 410 + t, outl, "cuda") for t in range(2)])
    n = x.shape[0]
    block = torch.empty(n * (16384 + 9216), dtype=torch.uint8, device="cuda")
    anc = block[:n * 16384].view(n, 128, 128)
    meta = block[n * 16384:].view(torch.float32).view(n, 2304)
    res = torch.empty_like(anc)
    L.lynx_encode_pages(x, L.Params(), anc, res, meta)
    a2, r2, m2 = L.lynx_encode_pages(x)
    torch.cuda.synchronize()
    assert torch.equal(anc, a2) and torch.equal(res, r2) and torch.equal(meta, m2)
    assert torch.equal(L.lynx_reconstruct(anc, None, meta), L.lynx_reconstruct(a2, None, m2))
    npph = n_tok // 256
    pt = torch.arange(n_heads * npph, dtype=torch.int32, device="cuda").view(1, n_heads, npph)
    ctx = torch.full((1,), n_tok, dtype=torch.int32, device="cuda")
    q = inputs.queries_torch((1, 1, 4 * n_heads, 128), 42, "cuda")
    vo = n_heads * npph
    o1, l1 = L.lynx_decode_attn(q, anc, None, meta, anc[vo:], None, meta[vo:], pt, ctx, n_heads)
    o2, l2 = L.lynx_decode_attn(q, a2, None, m2, a2[vo:], None, m2[vo:], pt, ctx, n_heads)
    torch.cuda.synchronize()
    L.lynx_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
