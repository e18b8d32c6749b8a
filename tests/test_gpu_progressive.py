"""Progressive (Anchor-first) transfer of an encoded cache between two sets of
device buffers through pinned host memory: every byte arrives unchanged, every
Anchor lands before any Residual, and a draft decode that waits only for the
Anchor events gives the same result as over the source buffers."""
import numpy as np
import pytest
import torch

from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L
from progressive_kv_quantization_gb300.progressive import ProgressiveTransfer

pytestmark = pytest.mark.gpu


def test_anchor_first_transfer_and_draft_on_the_anchor(cuda_device):
    n_layers, Hkv, npph = 4, 2, 8                   # per layer: K then V, Hkv heads x npph pages
    per = Hkv * npph
    out = inputs.outlier_pairs(Hkv, 90)
    x = torch.cat([inputs.kv_pages_torch(Hkv, 256 * npph, inputs.layer_seed(90, l, t), out, "cuda")
                   for l in range(n_layers) for t in range(2)])
    src = L.lynx_encode_pages(x)
    dst = tuple(torch.zeros_like(t) for t in src)
    layers = [(2 * l * per, 2 * (l + 1) * per) for l in range(n_layers)]
    tr = ProgressiveTransfer(layers).send(src, dst)

    # the consumer drafts on each layer once its Anchor has landed
    Hq = 4 * Hkv
    q = torch.from_numpy(inputs.queries_np((1, 1, Hq, 128), 91).view(np.int16)).view(torch.bfloat16).cuda()
    ctx = torch.tensor([256 * npph], dtype=torch.int32, device="cuda")
    consumer = torch.cuda.Stream()
    got, ref = [], []
    for l in range(n_layers):
        table = torch.tensor([[[2 * l * per + h * npph + p for p in range(npph)] for h in range(Hkv)]],
                             dtype=torch.int32, device="cuda")
        with torch.cuda.stream(consumer):
            consumer.wait_event(tr.anchor_ready[l])
            got.append(L.lynx_decode_attn(q, dst[0], None, dst[2], dst[0][per:], None, dst[2][per:], table, ctx,
                                          Hkv)[0])
        ref.append(L.lynx_decode_attn(q, src[0], None, src[2], src[0][per:], None, src[2][per:], table, ctx,
                                      Hkv)[0])
    torch.cuda.synchronize()
    L.lynx_device_status()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    for a, b in zip(src, dst):
        assert torch.equal(a, b)
    t_anchor, t_full = tr.times_ms()
    assert 0 < t_anchor <= tr.start.elapsed_time(tr.full_ready[0]) <= t_full


def test_encode_overlapped_transfer_chains_draft_and_verification(cuda_device):
    """encode_and_send: each layer is encoded and sent while the next one is
    encoded (Anchor + metadata on a high-priority stream, the Residual on a
    low-priority one).  On the receiving side the draft decode of layer l waits
    only for anchor_ready[l] and the T-token verification of layer l only for
    full_ready[l].  The received bytes equal a direct encode; the drafts equal
    the same decode over the sender's planes; the verifications match the
    float64 oracle over the oracle's own encoding of the same BF16 pages."""
    import math

    from oracle import attention as at
    from oracle import lynx_oracle as lo

    from lynx_testutil import EPS, check_attention

    n_layers, Hkv, npph, T = 3, 2, 4, 4
    per = Hkv * npph
    out = inputs.outlier_pairs(Hkv, 95)
    bits = [inputs.kv_pages_np(Hkv, 256 * npph, inputs.layer_seed(95, l, t), out)
            for l in range(n_layers) for t in range(2)]
    x_np = np.concatenate(bits)
    x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).cuda()
    n = x.shape[0]
    src = (torch.empty((n, 128, 128), dtype=torch.uint8, device="cuda"),
           torch.empty((n, 128, 128), dtype=torch.uint8, device="cuda"),
           torch.empty((n, L.META_FLOATS), dtype=torch.float32, device="cuda"))
    dst = tuple(torch.zeros_like(t) for t in src)
    layers = [(2 * l * per, 2 * (l + 1) * per) for l in range(n_layers)]
    tr = ProgressiveTransfer(layers)
    Hq = 4 * Hkv
    q1 = torch.from_numpy(inputs.queries_np((1, 1, Hq, 128), 96).view(np.int16)).view(torch.bfloat16).cuda()
    qv_np = inputs.queries_np((1, T, Hq, 128), 97)
    qv = torch.from_numpy(qv_np.view(np.int16)).view(torch.bfloat16).cuda()
    ctx = torch.tensor([256 * npph], dtype=torch.int32, device="cuda")
    table = torch.arange(per, dtype=torch.int32, device="cuda").view(1, Hkv, npph)
    producer, consumer = torch.cuda.Stream(), torch.cuda.Stream()
    tr.encode_and_send(x, src, dst, stream=producer)
    drafts, verifs = [], []
    for l, (a, _) in enumerate(layers):
        kv = lambda t: (t[a:], t[a + per:])
        with torch.cuda.stream(consumer):
            consumer.wait_event(tr.anchor_ready[l])
            (ka, va), (km, vm) = kv(dst[0]), kv(dst[2])
            drafts.append(L.lynx_decode_attn(q1, ka, None, km, va, None, vm, table, ctx, Hkv)[0])
            consumer.wait_event(tr.full_ready[l])
            (kr, vr) = kv(dst[1])
            verifs.append(L.lynx_decode_attn(qv, ka, kr, km, va, vr, vm, table, ctx, Hkv, causal=True))
    torch.cuda.synchronize()
    L.lynx_device_status()
    direct = L.lynx_encode_pages(x)
    for a_, b_ in zip(direct, dst):
        assert torch.equal(a_, b_)
    t_anchor, t_full = tr.times_ms()
    # every Anchor lands before any Residual; layer l's encode ends before its Anchor lands
    assert 0 < t_anchor <= min(tr.start.elapsed_time(e) for e in tr.full_ready) <= t_full
    for l in range(n_layers):
        assert tr.start.elapsed_time(tr.encoded[l]) <= tr.start.elapsed_time(tr.anchor_ready[l])
    for l, (a, _) in enumerate(layers):
        ref = L.lynx_decode_attn(q1, src[0][a:], None, src[2][a:], src[0][a + per:], None, src[2][a + per:],
                                 table, ctx, Hkv)[0]
        assert torch.equal(drafts[l], ref)
        oa, orr, om = lo.encode_pages(x_np[a:a + 2 * per], 100.0, EPS)
        kf = lo.reconstruct(oa[:per], orr[:per], om[:per], 100.0, EPS)
        vf = lo.reconstruct(oa[per:], orr[per:], om[per:], 100.0, EPS)
        ro, rl = at.decode_attention(lo.bf16_to_f32(qv_np).astype(np.float64), lambda ids: (kf[ids], vf[ids]),
                                     table.cpu().numpy(), np.array([256 * npph]), Hkv, 1 / math.sqrt(128), True)
        o, lse = verifs[l]
        check_attention(o.cpu().numpy(), lse.cpu().numpy(), ro, rl)
