"""lynx_decode_attn_noalloc: the decode attention for callers that cannot
allocate device memory (e.g. a connector plugin running inside a serving
engine's fixed memory budget, or a decode loop that must not call cudaMalloc
because it synchronises the device).  It uses the library's own static 8 MiB
scratch instead of a caller workspace.

Checked through the C ABI against lynx_decode_attn with a caller workspace, on
two calls in a row with different shapes and queries (the scratch keeps the
previous call's contents).  This file sorts last so that a run stopping at the
first failure has run every other test first; it also passes on its own in a
fresh process.
"""
import numpy as np
import pytest
import torch

from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L

from lynx_testutil import ATTN_TOL

pytestmark = pytest.mark.gpu


def _pools(Hkv, n_tok, seed):
    out = inputs.outlier_pairs(Hkv, seed)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
    k = L.lynx_encode_pages(dev(inputs.kv_pages_np(Hkv, n_tok, seed * 3 + 1, out)))
    v = L.lynx_encode_pages(dev(inputs.kv_pages_np(Hkv, n_tok, seed * 3 + 2, out)))
    return k, v


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    fin = np.isfinite(b)
    assert np.array_equal(fin, np.isfinite(a))
    err = np.abs(a[fin] - b[fin]) / np.maximum(1.0, np.abs(b[fin]))
    assert err.max() <= ATTN_TOL


def test_noalloc_matches_workspace_entry_point_twice(cuda_device):
    Hkv, Hq, n_tok = 8, 32, 4096
    (ka, kr, km), (va, vr, vm) = _pools(Hkv, n_tok, 1)
    npph = n_tok // 256
    calls = [
        # (B, T, full codes, causal, ctx lengths)
        (2, 1, False, False, [4096, 1000]),
        (3, 8, True, True, [4096, 2560, 300]),
    ]
    for i, (B, T, full, causal, ctx) in enumerate(calls):
        q = inputs.queries_torch((B, T, Hq, 128), 10 + i, "cuda")
        table = torch.stack([torch.stack([h * npph + torch.arange(npph, dtype=torch.int32) for h in range(Hkv)])
                             for _ in range(B)]).cuda()
        cl = torch.tensor(ctx, dtype=torch.int32, device="cuda")
        args = (q, ka, kr if full else None, km, va, vr if full else None, vm, table, cl, Hkv)
        o_ref, l_ref = L.lynx_decode_attn(*args, causal=causal)
        o, l = torch.empty_like(o_ref), torch.empty_like(l_ref)
        L.lynx_decode_attn_noalloc(*args, causal=causal, out=o, lse=l)   # warm-up: resolves the scratch
        torch.cuda.synchronize()
        free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        L.lynx_decode_attn_noalloc(*args, causal=causal, out=o, lse=l)
        torch.cuda.synchronize()
        # the call allocated nothing: neither the device's free memory nor torch's allocator moved
        assert torch.cuda.mem_get_info()[0] == free0 and torch.cuda.memory_allocated() == alloc0
        L.lynx_device_status()
        _close(o, o_ref)
        _close(l, l_ref)


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_device):
    # B=1024 sequences x 8 KV heads x 32 verification rows needs far more than 8 MiB
    B, T, Hq, Hkv, max_pages = 1024, 32, 32, 8, 512
    assert L.lynx_decode_attn_workspace_size(B, T, Hq, Hkv, 128, max_pages) > 8 << 20
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    lib = L.load()
    p = L.Params().c()
    import ctypes
    st = lib.lynx_decode_attn_noalloc(L._ptr(dummy), B, T, Hq, Hkv, 128, L._ptr(dummy), None, L._ptr(dummy),
                                      L._ptr(dummy), None, L._ptr(dummy), 1, L._ptr(dummy), max_pages,
                                      L._ptr(dummy), ctypes.byref(p), 0.088, 0, L._ptr(dummy), L._ptr(dummy),
                                      None)
    assert st == -4
    assert b"8 MiB" in lib.lynx_last_error()
