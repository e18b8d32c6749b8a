"""GPU parity of lynx_encode_split / lynx_reconstruct_split (the split stream at
other Anchor / Residual widths) against oracle/splits.py; the 4 + 4 split must
reproduce lynx_encode_pages / lynx_reconstruct byte for byte."""
import numpy as np
import pytest
import torch

from oracle import lynx_oracle as lo
from oracle import splits as sp
from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L

from lynx_testutil import CODE_EDGE, CODE_FRACTION, EPS, check_meta, check_recon, recon_bound

pytestmark = pytest.mark.gpu


def to_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _pages():
    return inputs.kv_pages_np(2, 768, 83, inputs.outlier_pairs(2, 83))


def test_four_four_split_is_the_split_stream(cuda_device):
    x = to_dev(_pages())
    a, r, m = L.lynx_encode_split(x, 4)
    a0, r0, m0 = L.lynx_encode_pages(x)
    assert torch.equal(a, a0) and torch.equal(r, r0) and torch.equal(m, m0)
    for res, res0 in ((None, None), (r, r0)):
        o = L.lynx_reconstruct_split(a, res, m, 4, out_dtype=torch.float32)
        o0 = L.lynx_reconstruct(a0, res0, m0, out_dtype=torch.float32)
        torch.cuda.synchronize()
        L.lynx_device_status()
        assert torch.equal(o, o0)


@pytest.mark.parametrize("A", [2, 3, 5, 6])
def test_split_widths_against_oracle(cuda_device, A):
    """Codes (via the 8-bit code they encode: equal except +-1 at rounding
    edges), metadata, Anchor-only and full reconstructions (float32 and BF16)
    against the oracle; the full reconstruction equals the 4 + 4 one bit for bit."""
    R = 8 - A
    bits = _pages()
    x = to_dev(bits)
    a, r, m = L.lynx_encode_split(x, A)
    oa, orr, om = sp.encode_pages_split(bits, A, 100.0, EPS)
    st = lo.run_stages(bits, 100.0, EPS)

    def q8(anc, res):
        qa = sp.unpack_bits(anc, A)
        V = np.where(qa < 0, -qa - 1, qa)
        I = (V << R) + (1 << (R - 1)) - 1 - sp.unpack_bits(res, R)
        return np.where(qa < 0, -I - 1, I)
    g, o = q8(a.cpu().numpy(), r.cpu().numpy()), q8(oa, orr)
    diff = g != o
    if diff.any():
        Yd = st.Y[diff]
        assert np.all(np.abs(Yd - np.floor(Yd) - 0.5) < CODE_EDGE)
    assert diff.mean() < CODE_FRACTION
    check_meta(m.cpu().numpy(), om)
    m_np = m.cpu().numpy()
    a_np, r_np = a.cpu().numpy(), r.cpu().numpy()
    for res, res_np in ((None, None), (r, r_np)):
        ref = sp.reconstruct_split(a_np, res_np, m_np, A, 100.0, EPS)
        for dt, is_bf16 in ((torch.float32, False), (torch.bfloat16, True)):
            out = L.lynx_reconstruct_split(a, res, m, A, out_dtype=dt)
            torch.cuda.synchronize()
            L.lynx_device_status()
            check_recon(out.float().cpu().numpy(), ref, recon_bound(m_np), is_bf16)
    a4, r4, m4 = L.lynx_encode_pages(x)
    assert torch.equal(L.lynx_reconstruct_split(a, r, m, A, out_dtype=torch.float32),
                       L.lynx_reconstruct(a4, r4, m4, out_dtype=torch.float32))
