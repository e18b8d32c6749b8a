"""GB300-native (sm_103a) Lynx hot path: split-stream KV quantiser, Anchor /
Anchor+Residual reconstruction and quantised-KV decode attention.

The compute lives in the CUDA library ``_build/liblynx.so`` (C ABI in
``include/lynx.h``); ``lynx`` is its thin Python binding and ``inputs`` the
seeded synthetic-input generators.  Importing the package does not load the
library; the first call does, and raises ``LynxError`` if it is missing.
"""
from .lynx import (  # noqa: F401
    LynxError,
    Params,
    lynx_attn_merge,
    lynx_encode_tokens,
    lynx_encode_variant,
    lynx_encode_split,
    lynx_reconstruct_split,
    lynx_reconstruct_variant,
    lynx_decode_attn_int4,
    lynx_decode_attn_uniform,
    lynx_split_nibbles,
    lynx_decode_attn,
    lynx_decode_attn_bf16,
    lynx_decode_attn_workspace_size,
    lynx_device_status,
    lynx_encode_pages,
    lynx_quantize_magnitudes,
    lynx_reconstruct,
    load,
)
