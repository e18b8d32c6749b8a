"""Thin Python binding of the Lynx C ABI (include/lynx.h).

Argument marshalling only: every function checks tensor types, allocates the
outputs the caller did not pass (torch device memory), and calls the entry
point of the same name in ``_build/liblynx.so`` on the current CUDA stream.
There is no fallback: if the library is missing or a call fails, a
``LynxError`` is raised.
"""
from __future__ import annotations

import ctypes
import functools
import math
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "liblynx.so")

H, P, C = 128, 256, 32
PLANE_BYTES = H * P // 2
META_FLOATS = 2 * H + 2 * H * (P // C)
OUT_BF16, OUT_F32 = 0, 1


class LynxError(RuntimeError):
    pass


class lynx_params_t(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("P", ctypes.c_int32), ("C", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("eps", ctypes.c_float)]


@dataclass(frozen=True)
class Params:
    alpha: float = 100.0
    eps: float = 1e-6
    H: int = H
    P: int = P
    C: int = C

    def c(self) -> lynx_params_t:
        return _params_struct(self.H, self.P, self.C, self.alpha, self.eps)


@functools.lru_cache(maxsize=64)
def _params_struct(H_, P_, C_, alpha, eps) -> lynx_params_t:
    """One C struct per parameter set (the library only reads it)."""
    return lynx_params_t(H_, P_, C_, alpha, eps)


_lib = None

# (name, restype, argtypes) of every exported entry point
_VP, _I64, _I32, _F32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_PP = ctypes.POINTER(lynx_params_t)
SIGNATURES = {
    "lynx_encode_pages": (_I32, [_VP, _I64, _PP, _VP, _VP, _VP, _VP]),
    "lynx_encode_pages_partial": (_I32, [_VP, _I64, _VP, _PP, _VP, _VP, _VP, _VP]),
    "lynx_encode_tokens": (_I32, [_VP, _I64, ctypes.c_int, _I64, _PP, _VP, _VP, _VP, _VP]),
    "lynx_reconstruct": (_I32, [_VP, _VP, _VP, _I64, _PP, _VP, _I32, _VP]),
    "lynx_quantize_magnitudes": (_I32, [_VP, _I64, _PP, _VP, _VP]),
    "lynx_decode_attn": (_I32, [_VP, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP,
                                _I64, _VP, _I32, _VP, _PP, _F32, _I32, _VP, _VP, _VP, _SZ, _VP]),
    "lynx_decode_attn_bf16": (_I32, [_VP, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _I64, _VP, _I32,
                                     _VP, _F32, _I32, _VP, _VP, _VP, _SZ, _VP]),
    "lynx_decode_attn_noalloc": (_I32, [_VP, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP,
                                        _I64, _VP, _I32, _VP, _PP, _F32, _I32, _VP, _VP, _VP]),
    "lynx_attn_merge": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _VP, _VP, _VP]),
    "lynx_encode_variant": (_I32, [_VP, _I64, _I32, _PP, _VP, _VP, _VP]),
    "lynx_decode_attn_uniform": (_I32, [_VP, _I32, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP,
                                        _I64, _VP, _I32, _VP, _F32, _I32, _VP, _VP, _VP, _SZ, _VP]),
    "lynx_split_nibbles": (_I32, [_VP, _I64, _VP, _VP, _VP]),
    "lynx_encode_split": (_I32, [_VP, _I64, _I32, _PP, _VP, _VP, _VP, _VP]),
    "lynx_reconstruct_split": (_I32, [_VP, _VP, _VP, _I64, _I32, _PP, _VP, _I32, _VP]),
    "lynx_reconstruct_variant": (_I32, [_VP, _VP, _I64, _I32, _PP, _VP, _I32, _VP]),
    "lynx_decode_attn_int4": (_I32, [_VP, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _VP, _VP, _I64, _VP, _I32,
                                     _VP, _PP, _F32, _I32, _VP, _VP, _VP, _SZ, _VP]),
    "lynx_decode_attn_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "lynx_device_status": (_I32, []),
    "lynx_test_inject_wait_timeout": (_I32, [_I32]),
    "lynx_status_string": (ctypes.c_char_p, [_I32]),
    "lynx_last_error": (ctypes.c_char_p, []),
    "lynx_version": (_I32, []),
}


def load(path: str = LIB_PATH):
    """Load liblynx.so (built by ``progressive_kv_quantization_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise LynxError(f"{path} is missing: build the CUDA library first "
                        "(python -m progressive_kv_quantization_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        lib = load()
        raise LynxError(f"{what}: {lib.lynx_status_string(status).decode()} "
                        f"({lib.lynx_last_error().decode()})")


def _ptr(t):
    # the argtypes are c_void_p, which takes the integer address directly
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device=None):
    """cudaStream_t of `stream`, or of torch's current stream on `device` (the
    tensor's device; the current device when None)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device() if device is None else device.index)
    return torch.cuda.current_stream(device).cuda_stream


def _need(t, dtype, name, device=None):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_contiguous():
        raise LynxError(f"{name} must be a contiguous {dtype} tensor")
    if not t.is_cuda:
        raise LynxError(f"{name} must live on a CUDA device")


def lynx_encode_pages(x, params: Params = Params(), anchor=None, residual=None, meta=None,
                      stream=None, valid_tokens=None):
    """Algorithm 1 on BF16 pages x[N, 128, 256] -> (anchor u8[N,128,128],
    residual u8[N,128,128], meta f32[N, 2304]).  valid_tokens (int32 [N] on the
    device, optional) selects lynx_encode_pages_partial: only the first
    valid_tokens[n] tokens of page n are valid."""
    _need(x, torch.bfloat16, "x")
    n = x.numel() // (H * P)
    if x.numel() != n * H * P:
        raise LynxError("x must hold whole 128 x 256 pages")
    dev = x.device
    anchor = anchor if anchor is not None else torch.empty((n, H, P // 2), dtype=torch.uint8, device=dev)
    residual = residual if residual is not None else torch.empty((n, H, P // 2), dtype=torch.uint8, device=dev)
    meta = meta if meta is not None else torch.empty((n, META_FLOATS), dtype=torch.float32, device=dev)
    for t, nm in ((anchor, "anchor"), (residual, "residual")):
        _need(t, torch.uint8, nm)
    _need(meta, torch.float32, "meta")
    if anchor.numel() < n * PLANE_BYTES or residual.numel() < n * PLANE_BYTES or meta.numel() < n * META_FLOATS:
        raise LynxError("output buffers too small")
    p = params.c()
    if valid_tokens is not None:
        _need(valid_tokens, torch.int32, "valid_tokens")
        if valid_tokens.numel() != n:
            raise LynxError("valid_tokens needs one count per page")
        _check(load().lynx_encode_pages_partial(_ptr(x), n, _ptr(valid_tokens), ctypes.byref(p), _ptr(anchor),
                                                _ptr(residual), _ptr(meta), _stream(stream)),
               "lynx_encode_pages_partial")
        return anchor, residual, meta
    _check(load().lynx_encode_pages(_ptr(x), n, ctypes.byref(p), _ptr(anchor), _ptr(residual),
                                    _ptr(meta), _stream(stream)), "lynx_encode_pages")
    return anchor, residual, meta


def lynx_encode_tokens(x, n_heads: int, params: Params = Params(), anchor=None, residual=None, meta=None,
                       stream=None):
    """Algorithm 1 on token-major KV (the layout of paged attention): x is a
    BF16 tensor whose first dimension is the token and whose row holds head h's
    128 channels at elements h*128 .. h*128 + 127 (e.g. [n_tokens, n_heads, 128],
    or a row-strided view of a wider buffer).  Returns the pages (n_heads *
    ceil(n_tokens / 256) of them, page h * n_pp + j = tokens 256 j .. of head h)
    as lynx_encode_pages does; each head's last page is encoded over its valid
    tokens."""
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or not x.is_cuda:
        raise LynxError("x must be a CUDA bfloat16 tensor")
    n_tokens = x.shape[0]
    inner = x[0].numel() if n_tokens > 0 else 0
    if n_tokens > 0 and (inner < n_heads * H or not x[0].is_contiguous()):
        raise LynxError("each token row must hold n_heads * 128 contiguous channels")
    stride = x.stride(0) if n_tokens > 0 else n_heads * H
    n_pp = (n_tokens + P - 1) // P
    n = n_heads * n_pp
    dev = x.device
    anchor = anchor if anchor is not None else torch.empty((n, H, P // 2), dtype=torch.uint8, device=dev)
    residual = residual if residual is not None else torch.empty((n, H, P // 2), dtype=torch.uint8, device=dev)
    meta = meta if meta is not None else torch.empty((n, META_FLOATS), dtype=torch.float32, device=dev)
    for t, nm in ((anchor, "anchor"), (residual, "residual")):
        _need(t, torch.uint8, nm)
    _need(meta, torch.float32, "meta")
    if anchor.numel() < n * PLANE_BYTES or residual.numel() < n * PLANE_BYTES or meta.numel() < n * META_FLOATS:
        raise LynxError("output buffers too small")
    p = params.c()
    _check(load().lynx_encode_tokens(_ptr(x), n_tokens, n_heads, stride, ctypes.byref(p), _ptr(anchor),
                                     _ptr(residual), _ptr(meta), _stream(stream)), "lynx_encode_tokens")
    return anchor, residual, meta


def lynx_quantize_magnitudes(a, params: Params = Params(), codes=None, stream=None):
    """Stage 3 alone: 7-bit magnitude codes (uint8) of float32 magnitudes a."""
    _need(a, torch.float32, "a")
    codes = codes if codes is not None else torch.empty(a.shape, dtype=torch.uint8, device=a.device)
    _need(codes, torch.uint8, "codes")
    p = params.c()
    _check(load().lynx_quantize_magnitudes(_ptr(a), a.numel(), ctypes.byref(p), _ptr(codes),
                                           _stream(stream)), "lynx_quantize_magnitudes")
    return codes


def lynx_reconstruct(anchor, residual, meta, params: Params = Params(), out=None,
                     out_dtype=torch.bfloat16, stream=None):
    """Anchor-only (residual=None) or full reconstruction -> out[N, 128, 256]."""
    _need(anchor, torch.uint8, "anchor")
    if residual is not None:
        _need(residual, torch.uint8, "residual")
    _need(meta, torch.float32, "meta")
    n = anchor.numel() // PLANE_BYTES
    code = {torch.bfloat16: OUT_BF16, torch.float32: OUT_F32}.get(out_dtype)
    if code is None:
        raise LynxError("out_dtype must be torch.bfloat16 or torch.float32")
    out = out if out is not None else torch.empty((n, H, P), dtype=out_dtype, device=anchor.device)
    _need(out, out_dtype, "out")
    p = params.c()
    _check(load().lynx_reconstruct(_ptr(anchor), _ptr(residual), _ptr(meta), n, ctypes.byref(p),
                                   _ptr(out), code, _stream(stream)), "lynx_reconstruct")
    return out


# single-precision variants (paper §6.1): name -> (LYNX_VARIANT_* value, code bytes per page, meta floats per page)
VARIANTS = {
    "lynx_int8": (1, H * P, META_FLOATS),
    "lynx_int4": (2, H * P // 2, META_FLOATS),
    "uniform_int8": (3, H * P, 2 * H),
    "uniform_int4": (4, H * P // 2, 2 * H),
}


def lynx_encode_variant(x, variant: str, params: Params = Params(), codes=None, meta=None, stream=None):
    """BF16 pages x[N, 128, 256] -> (codes u8[N, code bytes per page], meta f32[N, meta floats])
    of a single-precision variant: "lynx_int8", "lynx_int4", "uniform_int8" or
    "uniform_int4" (layouts in lynx.h)."""
    if variant not in VARIANTS:
        raise LynxError(f"unknown variant {variant!r}")
    code, cb, mf = VARIANTS[variant]
    _need(x, torch.bfloat16, "x")
    n = x.numel() // (H * P)
    if x.numel() != n * H * P:
        raise LynxError("x must hold whole 128 x 256 pages")
    codes = codes if codes is not None else torch.empty((n, cb), dtype=torch.uint8, device=x.device)
    meta = meta if meta is not None else torch.empty((n, mf), dtype=torch.float32, device=x.device)
    _need(codes, torch.uint8, "codes")
    _need(meta, torch.float32, "meta")
    if codes.numel() < n * cb or meta.numel() < n * mf:
        raise LynxError("output buffers too small")
    p = params.c()
    _check(load().lynx_encode_variant(_ptr(x), n, code, ctypes.byref(p), _ptr(codes), _ptr(meta),
                                      _stream(stream)), "lynx_encode_variant")
    return codes, meta


def lynx_reconstruct_variant(codes, meta, variant: str, params: Params = Params(), out=None,
                             out_dtype=torch.bfloat16, stream=None):
    """Dequantise a variant's codes and meta -> out[N, 128, 256]."""
    if variant not in VARIANTS:
        raise LynxError(f"unknown variant {variant!r}")
    code, cb, mf = VARIANTS[variant]
    _need(codes, torch.uint8, "codes")
    _need(meta, torch.float32, "meta")
    n = codes.numel() // cb
    if meta.numel() < n * mf:
        raise LynxError("meta too small")
    oc = {torch.bfloat16: OUT_BF16, torch.float32: OUT_F32}.get(out_dtype)
    if oc is None:
        raise LynxError("out_dtype must be torch.bfloat16 or torch.float32")
    out = out if out is not None else torch.empty((n, H, P), dtype=out_dtype, device=codes.device)
    _need(out, out_dtype, "out")
    p = params.c()
    _check(load().lynx_reconstruct_variant(_ptr(codes), _ptr(meta), n, code, ctypes.byref(p), _ptr(out), oc,
                                           _stream(stream)), "lynx_reconstruct_variant")
    return out


def lynx_encode_split(x, anchor_bits: int, params: Params = Params(), anchor=None, residual=None, meta=None,
                      stream=None):
    """The split stream with an A-bit Anchor (2..6): BF16 pages x[N, 128, 256] ->
    (anchor u8[N, 128, 32 A], residual u8[N, 128, 32 (8 - A)], meta f32[N, 2304])."""
    _need(x, torch.bfloat16, "x")
    n = x.numel() // (H * P)
    if x.numel() != n * H * P:
        raise LynxError("x must hold whole 128 x 256 pages")
    A, R = int(anchor_bits), 8 - int(anchor_bits)
    dev = x.device
    anchor = anchor if anchor is not None else torch.empty((n, H, 32 * A), dtype=torch.uint8, device=dev)
    residual = residual if residual is not None else torch.empty((n, H, 32 * R), dtype=torch.uint8, device=dev)
    meta = meta if meta is not None else torch.empty((n, META_FLOATS), dtype=torch.float32, device=dev)
    for t, nm, nb in ((anchor, "anchor", 32 * A), (residual, "residual", 32 * R)):
        _need(t, torch.uint8, nm)
        if t.numel() < n * H * nb:
            raise LynxError(f"{nm} too small")
    _need(meta, torch.float32, "meta")
    p = params.c()
    _check(load().lynx_encode_split(_ptr(x), n, A, ctypes.byref(p), _ptr(anchor), _ptr(residual), _ptr(meta),
                                    _stream(stream)), "lynx_encode_split")
    return anchor, residual, meta


def lynx_reconstruct_split(anchor, residual, meta, anchor_bits: int, params: Params = Params(), out=None,
                           out_dtype=torch.bfloat16, stream=None):
    """Anchor-only (residual=None) or full reconstruction of lynx_encode_split's planes."""
    _need(anchor, torch.uint8, "anchor")
    if residual is not None:
        _need(residual, torch.uint8, "residual")
    _need(meta, torch.float32, "meta")
    A = int(anchor_bits)
    n = anchor.numel() // (H * 32 * A)
    code = {torch.bfloat16: OUT_BF16, torch.float32: OUT_F32}.get(out_dtype)
    if code is None:
        raise LynxError("out_dtype must be torch.bfloat16 or torch.float32")
    out = out if out is not None else torch.empty((n, H, P), dtype=out_dtype, device=anchor.device)
    _need(out, out_dtype, "out")
    p = params.c()
    _check(load().lynx_reconstruct_split(_ptr(anchor), _ptr(residual), _ptr(meta), n, A, ctypes.byref(p),
                                         _ptr(out), code, _stream(stream)), "lynx_reconstruct_split")
    return out


def lynx_decode_attn_workspace_size(B, T, Hq, Hkv, head_dim, max_pages) -> int:
    return int(load().lynx_decode_attn_workspace_size(B, T, Hq, Hkv, head_dim, max_pages))


def _pool_pages(k_anc, k_res, k_meta, v_anc, v_res, v_meta) -> int:
    """Pages addressable in every pool passed (page ids must stay below it)."""
    for t, nm in ((k_anc, "k_anc"), (v_anc, "v_anc")):
        _need(t, torch.uint8, nm)
    for t, nm in ((k_meta, "k_meta"), (v_meta, "v_meta")):
        _need(t, torch.float32, nm)
    n = min(k_anc.numel(), v_anc.numel()) // PLANE_BYTES
    n = min(n, k_meta.numel() // META_FLOATS, v_meta.numel() // META_FLOATS)
    for t in (k_res, v_res):
        if t is not None:
            _need(t, torch.uint8, "residual pool")
            n = min(n, t.numel() // PLANE_BYTES)
    return n


def _decode_prep(q, page_table, ctx_len, n_kv_heads, out, lse, workspace):
    _need(q, torch.bfloat16, "q")
    if q.dim() != 4:
        raise LynxError("q must be [B, T, Hq, 128]")
    B, T, Hq, D = q.shape
    _need(page_table, torch.int32, "page_table")
    _need(ctx_len, torch.int32, "ctx_len")
    if page_table.dim() != 3 or page_table.shape[0] != B or page_table.shape[1] != n_kv_heads:
        raise LynxError("page_table must be [B, Hkv, max_pages]")
    max_pages = page_table.shape[2]
    dev = q.device
    out = out if out is not None else torch.empty((B, T, Hq, D), dtype=torch.float32, device=dev)
    lse = lse if lse is not None else torch.empty((B, T, Hq), dtype=torch.float32, device=dev)
    _need(out, torch.float32, "out")
    if workspace is None:
        ws_bytes = lynx_decode_attn_workspace_size(B, T, Hq, n_kv_heads, D, max_pages)
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    return B, T, Hq, D, max_pages, out, lse, workspace


def lynx_decode_attn(q, k_anc, k_res, k_meta, v_anc, v_res, v_meta, page_table, ctx_len,
                     n_kv_heads, params: Params = Params(), sm_scale=None, causal=False,
                     out=None, lse=None, workspace=None, stream=None):
    """Attention of q[B, T, Hq, 128] over packed K/V page pools (k_res = v_res =
    None: anchor-only draft KV).  Returns (out f32[B,T,Hq,128], lse f32[B,T,Hq])."""
    B, T, Hq, D, max_pages, out, lse, workspace = _decode_prep(q, page_table, ctx_len, n_kv_heads,
                                                               out, lse, workspace)
    n_pool = _pool_pages(k_anc, k_res, k_meta, v_anc, v_res, v_meta)
    scale = float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(D)
    p = params.c()
    _check(load().lynx_decode_attn(
        _ptr(q), B, T, Hq, n_kv_heads, D, _ptr(k_anc), _ptr(k_res), _ptr(k_meta), _ptr(v_anc),
        _ptr(v_res), _ptr(v_meta), n_pool, _ptr(page_table), max_pages, _ptr(ctx_len),
        ctypes.byref(p), scale, int(bool(causal)), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)), "lynx_decode_attn")
    return out, lse


def lynx_decode_attn_int4(q, k_codes, k_meta, v_codes, v_meta, page_table, ctx_len, n_kv_heads,
                          params: Params = Params(), sm_scale=None, causal=False, out=None, lse=None,
                          workspace=None, stream=None):
    """Attention of q over Lynx-INT4 page pools (lynx_encode_variant(..., "lynx_int4"))."""
    B, T, Hq, D, max_pages, out, lse, workspace = _decode_prep(q, page_table, ctx_len, n_kv_heads,
                                                               out, lse, workspace)
    n_pool = _pool_pages(k_codes.view(-1, H, P // 2), None, k_meta, v_codes.view(-1, H, P // 2), None, v_meta)
    scale = float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(D)
    p = params.c()
    _check(load().lynx_decode_attn_int4(
        _ptr(q), B, T, Hq, n_kv_heads, D, _ptr(k_codes), _ptr(k_meta), _ptr(v_codes), _ptr(v_meta), n_pool,
        _ptr(page_table), max_pages, _ptr(ctx_len), ctypes.byref(p), scale, int(bool(causal)), _ptr(out),
        _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
        "lynx_decode_attn_int4")
    return out, lse


def lynx_split_nibbles(codes, lo=None, hi=None, stream=None):
    """One-byte codes [n, 128, 256] (e.g. uniform INT8) -> (lo, hi) nibble planes
    [n, 128, 128]: token 2j in the low half of byte j, 2j + 1 in the high half."""
    _need(codes, torch.uint8, "codes")
    if codes.numel() % (H * P) != 0:
        raise LynxError("codes must hold rows of 256 bytes, 128 rows per page")
    n = codes.numel() // (H * P)
    lo = lo if lo is not None else torch.empty((n, H, P // 2), dtype=torch.uint8, device=codes.device)
    hi = hi if hi is not None else torch.empty((n, H, P // 2), dtype=torch.uint8, device=codes.device)
    for t, nm in ((lo, "lo"), (hi, "hi")):
        _need(t, torch.uint8, nm)
        if t.numel() < n * PLANE_BYTES:
            raise LynxError(f"{nm} too small")
    _check(load().lynx_split_nibbles(_ptr(codes), n * H, _ptr(lo), _ptr(hi), _stream(stream)), "lynx_split_nibbles")
    return lo, hi


def lynx_decode_attn_uniform(q, bits, k_lo, k_hi, k_meta, v_lo, v_hi, v_meta, page_table, ctx_len, n_kv_heads,
                             sm_scale=None, causal=False, out=None, lse=None, workspace=None, stream=None):
    """Attention of q over uniform INT-b page pools (lynx_encode_variant(...,
    "uniform_int4" / "uniform_int8")): bits 4 takes the packed codes as k_lo /
    v_lo (k_hi = v_hi = None); bits 8 the nibble planes of lynx_split_nibbles."""
    B, T, Hq, D, max_pages, out, lse, workspace = _decode_prep(q, page_table, ctx_len, n_kv_heads,
                                                               out, lse, workspace)
    for t, nm in ((k_lo, "k_lo"), (v_lo, "v_lo")):
        _need(t, torch.uint8, nm)
    for t, nm in ((k_meta, "k_meta"), (v_meta, "v_meta")):
        _need(t, torch.float32, nm)
    n_pool = min(k_lo.numel(), v_lo.numel()) // PLANE_BYTES
    n_pool = min(n_pool, k_meta.numel() // (2 * H), v_meta.numel() // (2 * H))
    for t in (k_hi, v_hi):
        if t is not None:
            _need(t, torch.uint8, "high-nibble pool")
            n_pool = min(n_pool, t.numel() // PLANE_BYTES)
    scale = float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(D)
    _check(load().lynx_decode_attn_uniform(
        _ptr(q), B, T, Hq, n_kv_heads, D, int(bits), _ptr(k_lo), _ptr(k_hi), _ptr(k_meta), _ptr(v_lo), _ptr(v_hi),
        _ptr(v_meta), n_pool, _ptr(page_table), max_pages, _ptr(ctx_len), scale, int(bool(causal)), _ptr(out),
        _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
        "lynx_decode_attn_uniform")
    return out, lse


def lynx_decode_attn_noalloc(q, k_anc, k_res, k_meta, v_anc, v_res, v_meta, page_table, ctx_len,
                             n_kv_heads, params: Params = Params(), sm_scale=None, causal=False,
                             out=None, lse=None, stream=None):
    """lynx_decode_attn without a workspace argument: the library's own 8 MiB
    static scratch is used, for callers that cannot allocate device memory."""
    _need(q, torch.bfloat16, "q")
    B, T, Hq, D = q.shape
    max_pages = page_table.shape[2]
    out = out if out is not None else torch.empty((B, T, Hq, D), dtype=torch.float32, device=q.device)
    lse = lse if lse is not None else torch.empty((B, T, Hq), dtype=torch.float32, device=q.device)
    n_pool = _pool_pages(k_anc, k_res, k_meta, v_anc, v_res, v_meta)
    scale = float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(D)
    p = params.c()
    _check(load().lynx_decode_attn_noalloc(
        _ptr(q), B, T, Hq, n_kv_heads, D, _ptr(k_anc), _ptr(k_res), _ptr(k_meta), _ptr(v_anc),
        _ptr(v_res), _ptr(v_meta), n_pool, _ptr(page_table), max_pages, _ptr(ctx_len),
        ctypes.byref(p), scale, int(bool(causal)), _ptr(out), _ptr(lse), _stream(stream)),
        "lynx_decode_attn_noalloc")
    return out, lse


def lynx_decode_attn_bf16(q, k_pages, v_pages, page_table, ctx_len, n_kv_heads, sm_scale=None,
                          causal=False, out=None, lse=None, workspace=None, stream=None):
    """The same attention over BF16 page pools k_pages/v_pages[n, 128, 256]."""
    B, T, Hq, D, max_pages, out, lse, workspace = _decode_prep(q, page_table, ctx_len, n_kv_heads,
                                                               out, lse, workspace)
    _need(k_pages, torch.bfloat16, "k_pages")
    _need(v_pages, torch.bfloat16, "v_pages")
    n_pool = min(k_pages.numel(), v_pages.numel()) // (H * P)
    scale = float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(D)
    _check(load().lynx_decode_attn_bf16(
        _ptr(q), B, T, Hq, n_kv_heads, D, _ptr(k_pages), _ptr(v_pages), n_pool, _ptr(page_table),
        max_pages, _ptr(ctx_len), scale, int(bool(causal)), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)), "lynx_decode_attn_bf16")
    return out, lse


def lynx_attn_merge(o_a, lse_a, o_b, lse_b, out=None, lse=None, stream=None):
    """Log-sum-exp merge of two attention results over disjoint key sets:
    o_a, o_b [..., 128] float32 and lse_a, lse_b [...] float32 (natural log)."""
    for t, nm in ((o_a, "o_a"), (o_b, "o_b")):
        _need(t, torch.float32, nm)
    for t, nm in ((lse_a, "lse_a"), (lse_b, "lse_b")):
        _need(t, torch.float32, nm)
    if o_a.shape != o_b.shape or lse_a.shape != lse_b.shape or tuple(o_a.shape[:-1]) != tuple(lse_a.shape):
        raise LynxError("o_a/o_b [..., D] and lse_a/lse_b [...] shapes disagree")
    out = out if out is not None else torch.empty_like(o_a)
    lse = lse if lse is not None else torch.empty_like(lse_a)
    _check(load().lynx_attn_merge(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), lse_a.numel(),
                                  o_a.shape[-1], _ptr(out), _ptr(lse), _stream(stream)), "lynx_attn_merge")
    return out, lse


def lynx_device_status():
    """Raise if a kernel recorded an error (synchronises the device)."""
    _check(load().lynx_device_status(), "lynx_device_status")
