"""GPU parity of lynx_encode_tokens, the encoder reading token-major KV (the
layout of paged attention): against the oracle's page encoding of the same
tokens, and byte for byte against lynx_encode_pages / lynx_encode_pages_partial
on the transposed pages at the size of a Llama-3-8B layer."""
import numpy as np
import pytest
import torch

from oracle import lynx_oracle as lo
from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L

from lynx_testutil import EPS, check_codes, check_meta

pytestmark = pytest.mark.gpu


def token_major(pages_bits: np.ndarray, n_heads: int, n_tokens: int, extra: int, rng) -> np.ndarray:
    """[n_tokens, n_heads * 128 + extra] rows: token t of head h from page
    h * n_pp + t // 256 of the given channel-major pages; the extra columns
    hold unrelated bits."""
    n_pp = pages_bits.shape[0] // n_heads
    rows = np.empty((n_tokens, n_heads * 128 + extra), dtype=np.uint16)
    for h in range(n_heads):
        head = np.concatenate([pages_bits[h * n_pp + j].T for j in range(n_pp)], axis=0)
        rows[:, h * 128:(h + 1) * 128] = head[:n_tokens]
    rows[:, n_heads * 128:] = rng.integers(0, 1 << 16, (n_tokens, extra), dtype=np.uint16)
    return rows


def to_dev(bits: np.ndarray):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("n_tokens", [1, 31, 300, 512, 700])
@pytest.mark.parametrize("layout", ["aligned", "unaligned"])
def test_token_major_parity_against_oracle(cuda_device, n_tokens, layout):
    """2 heads, token rows wider than the heads: codes and metadata against the
    oracle's encoding of the same tokens, for tails at and around chunk edges
    and for whole pages.  "aligned": 64 unrelated channels per row (a
    16-byte-aligned start and a stride of 320 elements, the TMA-staged kernel);
    "unaligned": the heads start one element into the row and the stride is
    259 elements (the kernel that reads global memory directly)."""
    rng = np.random.default_rng(n_tokens)
    n_heads = 2
    n_pp = -(-n_tokens // 256)
    pages = inputs.kv_pages_np(n_heads, 256 * n_pp, 70 + n_tokens, inputs.outlier_pairs(n_heads, 70))
    if layout == "aligned":
        rows = token_major(pages, n_heads, n_tokens, 64, rng)
        x = to_dev(rows)
    else:
        rows = token_major(pages, n_heads, n_tokens, 2, rng)
        wide = np.concatenate([rng.integers(0, 1 << 16, (n_tokens, 1), dtype=np.uint16), rows], axis=1)
        x = to_dev(wide)[:, 1:]
        assert x.stride(0) == 259 and x.data_ptr() % 16 != 0
    a, r, m = L.lynx_encode_tokens(x, n_heads)
    torch.cuda.synchronize()
    L.lynx_device_status()
    opages, valid = lo.pages_from_tokens(rows, n_heads)
    oa, orr, om, st = lo.encode_pages(opages, 100.0, EPS, return_stages=True, valid=valid)
    check_codes(a.cpu().numpy(), r.cpu().numpy(), oa, orr, st.Y)
    check_meta(m.cpu().numpy(), om)


def test_token_major_equals_page_encoder_at_layer_size(cuda_device):
    """One Llama-3-8B-shaped layer (8 KV heads x 16,384 tokens), K and V
    interleaved per token ([tokens][2][8][128], each read through a strided
    view): every page equals lynx_encode_pages on the channel-major pages; with
    100 tokens fewer, each head's last page equals lynx_encode_pages_partial."""
    dev = torch.device("cuda")
    n_heads, n_tok = 8, 16384
    outl = inputs.outlier_pairs(n_heads, 3)
    kp = inputs.kv_pages_torch(n_heads, n_tok, 31, outl, dev)   # [512, 128, 256]
    vp = inputs.kv_pages_torch(n_heads, n_tok, 32, outl, dev)

    def rows_of(p):   # [8 heads * 64 pages, 128, 256] -> [16384 tokens, 8, 128]
        return p.view(n_heads, n_tok // 256, 128, 256).permute(1, 3, 0, 2).reshape(n_tok, n_heads, 128)
    kv = torch.stack([rows_of(kp), rows_of(vp)], dim=1).contiguous()   # [tokens, 2, 8, 128]
    for t, pages in ((0, kp), (1, vp)):
        a, r, m = L.lynx_encode_tokens(kv[:, t], n_heads)
        ea, er, em = L.lynx_encode_pages(pages)
        torch.cuda.synchronize()
        assert torch.equal(a, ea) and torch.equal(r, er) and torch.equal(m, em)
    n_short = n_tok - 100
    a, r, m = L.lynx_encode_tokens(kv[:n_short, 0], n_heads)
    valid = torch.tensor(([256] * 63 + [156]) * n_heads, dtype=torch.int32, device=dev)
    ea, er, em = L.lynx_encode_pages(kp, valid_tokens=valid)
    torch.cuda.synchronize()
    L.lynx_device_status()
    assert torch.equal(a, ea) and torch.equal(r, er) and torch.equal(m, em)
