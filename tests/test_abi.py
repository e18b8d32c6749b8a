"""The C ABI without a GPU: the library builds, loads, exports every entry
point include/lynx.h declares, and rejects bad arguments before launching."""
import ctypes
import os
import re

import pytest

from progressive_kv_quantization_gb300 import lynx as L

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lynx.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lynx_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("lynx_encode_pages", "lynx_reconstruct", "lynx_decode_attn"):
        assert required in names


def test_library_exports_every_declared_symbol(lynx_lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lynx_lib, n), f"{n} declared in lynx.h but not exported"
        assert n in L.SIGNATURES, f"{n} has no binding signature"


def _p(**kw):
    d = dict(H=128, P=256, C=32, alpha=100.0, eps=1e-6)
    d.update(kw)
    return L.lynx_params_t(d["H"], d["P"], d["C"], d["alpha"], d["eps"])


def test_encode_argument_checks(lynx_lib):
    lib = lynx_lib
    buf = ctypes.create_string_buffer(64)
    aligned = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    odd = ctypes.c_void_p(aligned.value + 1)
    ok = _p()
    assert lib.lynx_encode_pages(aligned, 1, None, aligned, aligned, aligned, None) == -1
    assert lib.lynx_encode_pages(aligned, 1, ctypes.byref(_p(H=64)), aligned, aligned, aligned, None) == -2
    assert lib.lynx_encode_pages(aligned, 1, ctypes.byref(_p(C=16)), aligned, aligned, aligned, None) == -2
    assert lib.lynx_encode_pages(aligned, 1, ctypes.byref(_p(alpha=0.0)), aligned, aligned, aligned, None) == -2
    assert lib.lynx_encode_pages(aligned, 1, ctypes.byref(_p(eps=0.0)), aligned, aligned, aligned, None) == -2
    assert lib.lynx_encode_pages(aligned, -1, ctypes.byref(ok), aligned, aligned, aligned, None) == -1
    assert lib.lynx_encode_pages(None, 1, ctypes.byref(ok), aligned, aligned, aligned, None) == -1
    assert lib.lynx_encode_pages(odd, 1, ctypes.byref(ok), aligned, aligned, aligned, None) == -3
    assert lib.lynx_encode_pages(None, 0, ctypes.byref(ok), None, None, None, None) == 0
    assert b"16-byte" in (lib.lynx_encode_pages(odd, 1, ctypes.byref(ok), aligned, aligned, aligned, None)
                          and lib.lynx_last_error())


def test_reconstruct_and_decode_argument_checks(lynx_lib):
    lib = lynx_lib
    buf = ctypes.create_string_buffer(64)
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    ok = ctypes.byref(_p())
    assert lib.lynx_reconstruct(a, None, a, 1, ok, a, 7, None) == -1
    assert lib.lynx_reconstruct(a, None, a, 0, ok, a, 0, None) == 0
    # decode: T > 64, Hq not a multiple of Hkv, head_dim != 128, mixed residual pools
    args = lambda **kw: dict(dict(q=a, B=1, T=1, Hq=32, Hkv=8, D=128, kr=None, vr=None,
                                  ws=a, wsb=0), **kw)

    def call(**kw):
        x = args(**kw)
        return lib.lynx_decode_attn(x["q"], x["B"], x["T"], x["Hq"], x["Hkv"], x["D"], a, x["kr"], a,
                                    a, x["vr"], a, 4, a, 4, a, ok, 0.088, 0, a, a, x["ws"], x["wsb"], None)
    assert call(T=65) == -2
    assert call(T=64, Hq=64) == -2           # T * Hq/Hkv = 512 > 256
    assert call(Hq=30) == -1
    assert call(D=64) == -2
    assert call(kr=a) == -1
    assert call(ws=None) == -4
    assert lib.lynx_decode_attn_workspace_size(1, 1, 32, 8, 128, 64) > 0
    assert lib.lynx_decode_attn_workspace_size(1, 64, 32, 8, 128, 64) > 0
    assert lib.lynx_decode_attn_workspace_size(1, 65, 32, 8, 128, 64) == 0


def test_status_strings(lynx_lib):
    for code, name in ((0, b"LYNX_OK"), (-3, b"LYNX_ERR_ALIGNMENT"), (-6, b"LYNX_ERR_DEVICE")):
        assert lynx_lib.lynx_status_string(code) == name
    assert lynx_lib.lynx_version() >= 100


def test_row_limit_merge_and_partial_argument_checks(lynx_lib):
    lib = lynx_lib
    buf = ctypes.create_string_buffer(64)
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    odd = ctypes.c_void_p(a.value + 4)
    ok = ctypes.byref(_p())
    # more than 256 query rows per KV head (T * Hq / Hkv = 32 * 9)
    assert lib.lynx_decode_attn(a, 1, 32, 72, 8, 128, a, None, a, a, None, a, 4, a, 4, a, ok, 0.088, 0,
                                a, a, a, 0, None) == -2
    # merge: negative rows, head_dim, alignment, empty
    assert lib.lynx_attn_merge(a, a, a, a, -1, 128, a, a, None) == -1
    assert lib.lynx_attn_merge(a, a, a, a, 4, 64, a, a, None) == -2
    assert lib.lynx_attn_merge(a, a, odd, a, 4, 128, a, a, None) == -3
    assert lib.lynx_attn_merge(a, a, a, a, 0, 128, a, a, None) == 0
    assert lib.lynx_attn_merge(None, a, a, a, 4, 128, a, a, None) == -1
    # partial encode: the valid counts are required, and must be aligned
    assert lib.lynx_encode_pages_partial(a, 1, None, ok, a, a, a, None) == -1
    assert lib.lynx_encode_pages_partial(a, 1, odd, ok, a, a, a, None) == -3
    assert lib.lynx_encode_pages_partial(a, 0, None, ok, a, a, a, None) == 0


def test_token_major_encode_argument_checks(lynx_lib):
    lib = lynx_lib
    buf = ctypes.create_string_buffer(64)
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    odd = ctypes.c_void_p(a.value + 1)
    ok = ctypes.byref(_p())
    # token_stride below n_heads * 128, negative counts, NULL, odd x, misaligned outputs, no work
    assert lib.lynx_encode_tokens(a, 300, 2, 255, ok, a, a, a, None) == -1
    assert lib.lynx_encode_tokens(a, -1, 2, 256, ok, a, a, a, None) == -1
    assert lib.lynx_encode_tokens(None, 300, 2, 256, ok, a, a, a, None) == -1
    assert lib.lynx_encode_tokens(odd, 300, 2, 256, ok, a, a, a, None) == -3
    assert lib.lynx_encode_tokens(a, 300, 2, 256, ok, ctypes.c_void_p(a.value + 4), a, a, None) == -3
    assert lib.lynx_encode_tokens(a, 0, 2, 256, ok, None, None, None, None) == 0
    assert lib.lynx_encode_tokens(a, 300, 0, 0, ok, None, None, None, None) == 0
    assert lib.lynx_encode_tokens(a, 300, 2, 256, ctypes.byref(_p(alpha=0.0)), a, a, a, None) == -2


def test_variant_argument_checks(lynx_lib):
    lib = lynx_lib
    buf = ctypes.create_string_buffer(64)
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    odd = ctypes.c_void_p(a.value + 4)
    ok = ctypes.byref(_p())
    for v in (0, 5):   # unknown variants
        assert lib.lynx_encode_variant(a, 1, v, ok, a, a, None) == -1
        assert lib.lynx_reconstruct_variant(a, a, 1, v, ok, a, 0, None) == -1
    assert lib.lynx_encode_variant(a, -1, 3, ok, a, a, None) == -1
    assert lib.lynx_encode_variant(odd, 1, 3, ok, a, a, None) == -3
    assert lib.lynx_encode_variant(a, 0, 2, ok, None, None, None) == 0
    assert lib.lynx_encode_variant(a, 1, 2, ctypes.byref(_p(alpha=0.0)), a, a, None) == -2
    # uniform variants do not read params
    assert lib.lynx_encode_variant(a, 0, 4, None, None, None, None) == 0
    assert lib.lynx_reconstruct_variant(a, a, 1, 1, ok, a, 7, None) == -1
    assert lib.lynx_reconstruct_variant(None, a, 1, 4, ok, a, 0, None) == -1


def test_split_argument_checks(lynx_lib):
    lib = lynx_lib
    buf = ctypes.create_string_buffer(64)
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    ok = ctypes.byref(_p())
    for bits in (1, 7):
        assert lib.lynx_encode_split(a, 1, bits, ok, a, a, a, None) == -2
        assert lib.lynx_reconstruct_split(a, a, a, 1, bits, ok, a, 0, None) == -2
    assert lib.lynx_encode_split(a, -1, 3, ok, a, a, a, None) == -1
    assert lib.lynx_encode_split(a, 0, 3, ok, None, None, None, None) == 0
    assert lib.lynx_encode_split(ctypes.c_void_p(a.value + 2), 1, 3, ok, a, a, a, None) == -3
    assert lib.lynx_reconstruct_split(a, None, a, 1, 3, ok, a, 9, None) == -1


def test_uniform_decode_and_nibble_split_argument_checks(lynx_lib):
    lib = lynx_lib
    buf = ctypes.create_string_buffer(64)
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    odd = ctypes.c_void_p(a.value + 4)

    def call(bits, k_hi=None, v_hi=None, k_lo=a, T=1):
        return lib.lynx_decode_attn_uniform(a, 1, T, 32, 8, 128, bits, k_lo, k_hi, a, a, v_hi, a, 4, a, 4, a,
                                            0.088, 0, a, a, a, 0, None)
    assert call(6) == -1                     # bits other than 4 and 8
    assert call(8) == -1                     # bits 8 without the high-nibble planes
    assert call(4, k_hi=a, v_hi=a) == -1     # bits 4 with them
    assert call(4, k_lo=None) == -1
    assert call(4, k_lo=odd) == -3
    assert call(4, T=65) == -2               # shape checks as lynx_decode_attn
    assert call(4) == -4                     # no workspace
    assert lib.lynx_split_nibbles(a, -1, a, a, None) == -1
    assert lib.lynx_split_nibbles(a, 0, None, None, None) == 0
    assert lib.lynx_split_nibbles(None, 1, a, a, None) == -1
    assert lib.lynx_split_nibbles(odd, 1, a, a, None) == -3
