"""A bounded wait that runs out, on the GPU, without a fault: the test hook
lynx_test_inject_wait_timeout makes the producer of every CTA skip the copy of
its first V page and shortens every wait to 1 ms.  The call must return, the
device error word must say that a wait gave up, and the next, normal call must
give exactly the result it gives without the fault (the kernel drained its
copies and freed its tensor memory).  Covers the draft kernel (anchor, T = 1),
the narrow kernel (full codes, T = 1; uniform INT4), the verification
kernel with 16-row register tiles (T = 4) and 32-row tensor-memory tiles
(T = 8), the BF16 decode kernel (8- and 16-row tiles), the staged
reconstruction (Anchor only and full codes) and the TMA-staged token-major
encoder."""
import numpy as np
import pytest
import torch

from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pools(cuda_device):
    Hkv, n_tok = 2, 16 * 256
    out = inputs.outlier_pairs(Hkv, 70)
    k = inputs.kv_pages_torch(Hkv, n_tok, 71, out, "cuda")
    v = inputs.kv_pages_torch(Hkv, n_tok, 72, out, "cuda")
    ka, kr, km = L.lynx_encode_pages(k)
    va, vr, vm = L.lynx_encode_pages(v)
    uk, um = L.lynx_encode_variant(k, "uniform_int4")
    uv, uvm = L.lynx_encode_variant(v, "uniform_int4")
    table = torch.arange(Hkv * 16, dtype=torch.int32, device="cuda").view(1, Hkv, 16)
    return dict(Hkv=Hkv, k=(ka, kr, km), v=(va, vr, vm), u=(uk, um, uv, uvm), kb=k, vb=v, table=table,
                ctx=torch.tensor([n_tok], dtype=torch.int32, device="cuda"))


def _call(p, mode, T):
    Hkv = p["Hkv"]
    q = inputs.queries_torch((1, T, 4 * Hkv, 128), 73 + T, "cuda")
    ka, kr, km = p["k"]
    va, vr, vm = p["v"]
    if mode == "bf16":
        return L.lynx_decode_attn_bf16(q, p["kb"], p["vb"], p["table"], p["ctx"], Hkv, causal=T > 1)
    if mode == "uniform4":
        uk, um, uv, uvm = p["u"]
        return L.lynx_decode_attn_uniform(q, 4, uk.view(-1, 128, 128), None, um, uv.view(-1, 128, 128), None, uvm,
                                          p["table"], p["ctx"], Hkv, causal=T > 1)
    full = mode == "full"
    return L.lynx_decode_attn(q, ka, kr if full else None, km, va, vr if full else None, vm, p["table"], p["ctx"],
                              Hkv, causal=T > 1)


@pytest.mark.parametrize("mode,T", [("anchor", 1), ("full", 1), ("uniform4", 1), ("full", 4), ("full", 8),
                                    ("anchor", 8), ("bf16", 1), ("bf16", 8)])
def test_wait_that_runs_out_is_reported_and_the_context_recovers(pools, mode, T):
    o_ref, l_ref = _call(pools, mode, T)
    torch.cuda.synchronize()
    L.lynx_device_status()
    lib = L.load()
    assert lib.lynx_test_inject_wait_timeout(1) == 0
    _call(pools, mode, T)
    torch.cuda.synchronize()
    with pytest.raises(L.LynxError, match="error word = 1"):
        L.lynx_device_status()
    L.lynx_device_status()       # read and cleared
    for _ in range(2):           # the hook fired once; later calls are normal and exact
        o, l = _call(pools, mode, T)
        torch.cuda.synchronize()
        L.lynx_device_status()
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


@pytest.mark.parametrize("full", [False, True])
def test_reconstruct_wait_that_runs_out_is_reported_and_the_context_recovers(pools, full):
    """The staged reconstruction: with the hook armed every CTA's producer skips
    its first page, the consumers' 1 ms waits run out, the error word is set;
    the next calls are normal and bit-identical to a call before the fault."""
    ka, kr, km = pools["k"]
    res = kr if full else None
    ref = L.lynx_reconstruct(ka, res, km)
    torch.cuda.synchronize()
    L.lynx_device_status()
    lib = L.load()
    assert lib.lynx_test_inject_wait_timeout(1) == 0
    L.lynx_reconstruct(ka, res, km)
    torch.cuda.synchronize()
    with pytest.raises(L.LynxError, match="error word = 1"):
        L.lynx_device_status()
    L.lynx_device_status()       # read and cleared
    for _ in range(2):
        out = L.lynx_reconstruct(ka, res, km)
        torch.cuda.synchronize()
        L.lynx_device_status()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_token_encoder_wait_that_runs_out_is_reported_and_the_context_recovers(cuda_device):
    """The TMA-staged token-major encoder (600 tokens of 3 heads: full pages
    and a partial last page, two launches): with the hook armed every CTA skips
    its first item's copy; the error word is set; later calls are exact."""
    n_heads, n_tok = 3, 600
    xt = inputs.queries_torch((n_tok, n_heads * 128), 77, "cuda")
    ref = [t.clone() for t in L.lynx_encode_tokens(xt, n_heads)]
    torch.cuda.synchronize()
    L.lynx_device_status()
    lib = L.load()
    assert lib.lynx_test_inject_wait_timeout(1) == 0
    L.lynx_encode_tokens(xt, n_heads)
    torch.cuda.synchronize()
    with pytest.raises(L.LynxError, match="error word = 1"):
        L.lynx_device_status()
    L.lynx_device_status()       # read and cleared
    for _ in range(2):
        got = L.lynx_encode_tokens(xt, n_heads)
        torch.cuda.synchronize()
        L.lynx_device_status()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_hook_rejects_negative_counts(cuda_device):
    lib = L.load()
    assert lib.lynx_test_inject_wait_timeout(-1) == -1
    assert lib.lynx_test_inject_wait_timeout(0) == 0
