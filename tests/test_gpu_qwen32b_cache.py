"""Parity on the Qwen-32B-shaped 64-layer cache at its full size, in the launch
configurations the benchmark times (whole-cache calls over 65,536 pages).

The cache is the benchmark's (seeded, generated on the device, encoded by the
GPU encoder); the planes and metadata of layers 0, 31 and 63 and of 256
sampled pages are then replaced by the oracle's own encoding of the same BF16
pages, so every compared output is computed from oracle inputs:

  * both reconstructions (BF16 out) of the whole cache in one launch, checked
    on the 256 sampled pages;
  * the B = 8 draft decode over the whole cache (512 sequences, sequence s of
    layer l reading layer (l + s) mod 64 through its page table), checked on
    every sequence that reads layer 0, 31 or 63;
  * the B = 1 draft decode and the T = 8 causal verification over the full
    codes (64 sequences, one per layer), checked on layers 0, 31 and 63.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as at
from oracle import lynx_oracle as lo
from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L

from lynx_testutil import EPS, check_attention, check_recon, recon_bound

pytestmark = pytest.mark.gpu

N_LAYERS, HKV, HQ, N_TOK = 64, 8, 32, 16384
NPPH = N_TOK // 256
PER = HKV * NPPH                 # pages per tensor per layer
LAYERS = (0, 31, 63)


@pytest.fixture(scope="module")
def cache(cuda_device):
    outl = inputs.outlier_pairs(HKV, 0)
    n = 2 * N_LAYERS * PER
    x = torch.empty((n, 128, 256), dtype=torch.bfloat16, device="cuda")
    for layer in range(N_LAYERS):
        for t in range(2):
            i = (2 * layer + t) * PER
            x[i:i + PER] = inputs.kv_pages_torch(HKV, N_TOK, inputs.layer_seed(0, layer, t), outl, "cuda")
    a, r, m = L.lynx_encode_pages(x)
    sample = np.sort(np.random.default_rng(11).choice(n, 256, replace=False))
    ids = np.concatenate([np.arange(2 * l * PER, 2 * (l + 1) * PER) for l in LAYERS] + [sample])
    ids = np.unique(ids)
    ti = torch.from_numpy(ids).cuda()
    bits = x[ti].view(torch.int16).cpu().numpy().view(np.uint16)
    oa, orr, om = lo.encode_pages(bits, 100.0, EPS)
    a[ti] = torch.from_numpy(oa).cuda()
    r[ti] = torch.from_numpy(orr).cuda()
    m[ti] = torch.from_numpy(om).cuda()
    pos = {int(p): k for k, p in enumerate(ids)}
    torch.cuda.synchronize()
    L.lynx_device_status()
    return dict(x=x, a=a, r=r, m=m, sample=sample, oa=oa, orr=orr, om=om, pos=pos)


def _oracle_layer(c, layer, full):
    """float64 dequantised K and V pages [PER, 128, 256] of one layer from the oracle's planes."""
    k = [c["pos"][p] for p in range(2 * layer * PER, (2 * layer + 1) * PER)]
    v = [c["pos"][p] for p in range(2 * layer * PER + PER, 2 * (layer + 1) * PER)]
    rec = lambda idx: lo.reconstruct(c["oa"][idx], c["orr"][idx] if full else None, c["om"][idx], 100.0, EPS)
    return rec(k), rec(v)


def _table(B, layer_of):
    t = np.empty((B, HKV, NPPH), dtype=np.int32)
    for b in range(B):
        for h in range(HKV):
            t[b, h] = 2 * layer_of(b) * PER + h * NPPH + np.arange(NPPH)
    return t


def test_reconstructions_of_the_whole_cache_sampled(cache):
    c = cache
    idx = [c["pos"][int(p)] for p in c["sample"]]
    ti = torch.from_numpy(c["sample"]).cuda()
    for full in (False, True):
        out = L.lynx_reconstruct(c["a"], c["r"] if full else None, c["m"], out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        got = out[ti].float().cpu().numpy()
        ref = lo.reconstruct(c["oa"][idx], c["orr"][idx] if full else None, c["om"][idx], 100.0, EPS)
        check_recon(got, ref, recon_bound(c["om"][idx]), True)
        del out


@pytest.mark.parametrize("B", [1, 8])
def test_draft_decode_over_the_whole_cache(cache, B):
    c = cache
    n_seq = B * N_LAYERS
    layer_of = (lambda s: s) if B == 1 else (lambda s: (s // 8 + s % 8) % N_LAYERS)
    table = _table(n_seq, layer_of)
    q_bits = inputs.queries_np((n_seq, 1, HQ, 128), 20 + B)
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    ctx = torch.full((n_seq,), N_TOK, dtype=torch.int32, device="cuda")
    kA, vA, kM, vM = c["a"], c["a"][PER:], c["m"], c["m"][PER:]
    o, lse = L.lynx_decode_attn(q, kA, None, kM, vA, None, vM, torch.from_numpy(table).cuda(), ctx, HKV)
    torch.cuda.synchronize()
    L.lynx_device_status()
    o, lse = o.cpu().numpy(), lse.cpu().numpy()
    qf = lo.bf16_to_f32(q_bits).astype(np.float64)
    scale = 1 / math.sqrt(128)
    for layer in LAYERS:
        kd, vd = _oracle_layer(c, layer, False)
        seqs = [s for s in range(n_seq) if layer_of(s) == layer]
        local = np.arange(PER, dtype=np.int32).reshape(1, HKV, NPPH)
        for s in seqs:
            ro, rl = at.decode_attention(qf[s:s + 1], lambda ids: (kd[ids], vd[ids]), local, np.array([N_TOK]),
                                         HKV, scale, False)
            check_attention(o[s:s + 1], lse[s:s + 1], ro, rl)


def test_verification_over_the_whole_cache(cache):
    c = cache
    T = 8
    table = _table(N_LAYERS, lambda s: s)
    q_bits = inputs.queries_np((N_LAYERS, T, HQ, 128), 31)
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    ctx = torch.full((N_LAYERS,), N_TOK, dtype=torch.int32, device="cuda")
    kA, vA, kR, vR, kM, vM = c["a"], c["a"][PER:], c["r"], c["r"][PER:], c["m"], c["m"][PER:]
    o, lse = L.lynx_decode_attn(q, kA, kR, kM, vA, vR, vM, torch.from_numpy(table).cuda(), ctx, HKV, causal=True)
    torch.cuda.synchronize()
    L.lynx_device_status()
    o, lse = o.cpu().numpy(), lse.cpu().numpy()
    qf = lo.bf16_to_f32(q_bits).astype(np.float64)
    local = np.arange(PER, dtype=np.int32).reshape(1, HKV, NPPH)
    for layer in LAYERS:
        kd, vd = _oracle_layer(c, layer, True)
        ro, rl = at.decode_attention(qf[layer:layer + 1], lambda ids: (kd[ids], vd[ids]), local,
                                     np.array([N_TOK]), HKV, 1 / math.sqrt(128), True)
        check_attention(o[layer:layer + 1], lse[layer:layer + 1], ro, rl)
