"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and lays them out; it holds none of the
quantiser's or the attention's arithmetic.  Both the CUDA path and the CPU
oracle receive the BF16 bit patterns it produces, so a parity test compares the
two on identical inputs.

Distribution (stand-in for the KV caches of the paper's workloads -- LLaMA-3.1-8B,
Qwen3-32B and Qwen3-235B-A22B on MMLU-Pro / Needle / QMSum -- which are not
available here; Lynx paper, §3.2 and Figures 4-5 describe the structure being
imitated: per-channel offsets, a few outlier channels about 100x larger, and a
sharp Laplacian-like spread around each channel's centre):

    x[h, c, t] = s[h, c] * (o[h, c] + lam[h, c, t])
    o   ~ N(0, 1)             one offset per (head, channel)
    lam ~ Laplace(0, 0.1)     scale parameter b = 0.1
    s   = 100 on outlier (head, channel) pairs, else 1

rounded to nearest-even BF16.  Queries are N(0, 1) rounded to BF16.

KV page layout (the layout every entry point of the library consumes): one page
is one KV head's 128 channels x 256 tokens, channel-major, i.e. a page is a
[128][256] BF16 array whose rows are the channels.  A head with L tokens owns
L/256 consecutive pages.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

H_CH = 128      # channels per page (one KV head's head_dim)
P_TOK = 256     # tokens per page
C_CHUNK = 32    # tokens per chunk


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest BF16 (ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def outlier_pairs(n_heads: int, seed: int, count: int | None = None) -> np.ndarray:
    """Outlier (head, channel) pairs as a boolean [n_heads, 128] mask.

    ``count`` defaults to round(1% of the head x channel pairs).  The single-page
    case passes ``count=4`` with one head.  The set depends only on the seed, so
    K and V and every layer of a multi-layer cache share it.
    """
    if count is None:
        count = int(round(0.01 * n_heads * H_CH))
    rng = np.random.default_rng(seed)
    idx = rng.choice(n_heads * H_CH, size=count, replace=False)
    mask = np.zeros(n_heads * H_CH, dtype=bool)
    mask[idx] = True
    return mask.reshape(n_heads, H_CH)


def kv_pages_np(n_heads: int, n_tokens: int, seed: int, outliers: np.ndarray,
                scale_outlier: float = 100.0, lap_b: float = 0.1) -> np.ndarray:
    """Host generator: BF16 bits of one KV tensor as pages [n_heads*n_tokens/256, 128, 256]."""
    assert n_tokens % P_TOK == 0
    rng = np.random.default_rng(seed)
    o = rng.standard_normal((n_heads, H_CH)).astype(np.float32)
    lam = rng.laplace(0.0, lap_b, size=(n_heads, H_CH, n_tokens)).astype(np.float32)
    s = np.where(outliers, np.float32(scale_outlier), np.float32(1.0)).astype(np.float32)
    x = s[:, :, None] * (o[:, :, None] + lam)
    npph = n_tokens // P_TOK
    pages = x.reshape(n_heads, H_CH, npph, P_TOK).transpose(0, 2, 1, 3)
    return f32_to_bf16_bits(np.ascontiguousarray(pages)).reshape(n_heads * npph, H_CH, P_TOK)


def queries_np(shape: tuple, seed: int) -> np.ndarray:
    """BF16 bits of N(0, 1) queries with the given shape (e.g. [B, T, Hq, 128])."""
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))


def kv_pages_torch(n_heads: int, n_tokens: int, seed: int, outliers_mask, device,
                   scale_outlier: float = 100.0, lap_b: float = 0.1):
    """Device generator for the large caches: returns a torch.bfloat16 tensor
    [n_heads*n_tokens/256, 128, 256] built on ``device`` from a seeded
    ``torch.Generator`` (Laplace drawn by inverse CDF from uniforms)."""
    import torch
    assert n_tokens % P_TOK == 0
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    npph = n_tokens // P_TOK
    o = torch.randn((n_heads, 1, H_CH, 1), generator=g, device=device, dtype=torch.float32)
    u = torch.rand((n_heads, npph, H_CH, P_TOK), generator=g, device=device,
                   dtype=torch.float32) - 0.5
    lam = -lap_b * torch.sign(u) * torch.log1p(-2.0 * u.abs().clamp(max=0.4999999))
    m = torch.as_tensor(np.asarray(outliers_mask), device=device)
    s = torch.where(m, torch.tensor(scale_outlier, device=device),
                    torch.tensor(1.0, device=device)).to(torch.float32)
    x = s.view(n_heads, 1, H_CH, 1) * (o + lam)
    return x.to(torch.bfloat16).reshape(n_heads * npph, H_CH, P_TOK)


def queries_torch(shape: tuple, seed: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def kv_bytes_bf16(n_layers: int, n_kv_heads: int, head_dim: int, n_tokens: int) -> int:
    """BF16 KV-cache size in bytes for K and V (2 bytes per element)."""
    return 2 * n_layers * n_kv_heads * head_dim * n_tokens * 2


@dataclass(frozen=True)
class Workload:
    """Shape of one of the synthetic workloads."""
    name: str
    n_layers: int
    n_kv_heads: int
    n_tokens: int
    n_q_heads: int

    @property
    def pages_per_head(self) -> int:
        return self.n_tokens // P_TOK

    @property
    def pages_per_tensor_layer(self) -> int:
        return self.n_kv_heads * self.pages_per_head

    @property
    def bf16_bytes(self) -> int:
        return kv_bytes_bf16(self.n_layers, self.n_kv_heads, H_CH, self.n_tokens)


SINGLE_PAGE = Workload("single KV page 128x256", 1, 1, 256, 1)
LLAMA8B_LAYER = Workload("Llama-3-8B-shaped layer: 8 KV heads x 128 x 16384 tokens", 1, 8, 16384, 32)
QWEN32B_CACHE = Workload("Qwen-32B-shaped cache: 64 layers x 8 KV heads x 128 x 16384 tokens", 64, 8, 16384, 32)
QWEN235B_CACHE = Workload("Qwen3-235B-A22B-shaped cache: 94 layers x 4 KV heads x 128 x 131072 tokens",
                          94, 4, 131072, 16)


def layer_seed(seed: int, layer: int, tensor: int) -> int:
    """Seed of one (layer, K-or-V) tensor of a multi-layer cache."""
    return seed * 1000 + 2 * layer + tensor


def pages_needed(n_tokens: int) -> int:
    return math.ceil(n_tokens / P_TOK)
