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
