"""GPU parity of lynx_attn_merge: attention over a union of two disjoint key
sets equals the log-sum-exp merge of the attention over each set.  Checked
against the float64 oracle's attention over the union, alone and as the paper's
verification pass needs it: the T draft tokens attend to the packed cache
(lynx_decode_attn) and to their own uncompressed K and V (a BF16 tail page,
lynx_decode_attn_bf16 with causal masking), merged."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as at
from oracle import lynx_oracle as lo
from progressive_kv_quantization_gb300 import inputs
from progressive_kv_quantization_gb300 import lynx as L

from lynx_testutil import EPS, check_attention

pytestmark = pytest.mark.gpu


def test_merge_equals_attention_over_the_union(cuda_device):
    rng = np.random.default_rng(3)
    R, La, Lb, D = 40, 300, 77, 128
    q = rng.standard_normal((R, D))
    ka, va = rng.standard_normal((La, D)) * 2, rng.standard_normal((La, D))
    kb, vb = rng.standard_normal((Lb, D)) * 2, rng.standard_normal((Lb, D))
    # per-row visible counts in each set; rows 0-2 see nothing in A, B, or either
    na = rng.integers(1, La + 1, R)
    nb = rng.integers(1, Lb + 1, R)
    na[0], nb[1], na[2], nb[2] = 0, 0, 0, 0
    s = 1 / math.sqrt(D)
    oa, la = at.attention_rows(q, ka, va, s, na)
    ob, lb = at.attention_rows(q, kb, vb, s, nb)
    k = np.concatenate([ka, kb])
    v = np.concatenate([va, vb])
    ou, lu = [], []
    for r in range(R):                               # union: A's first na keys and B's first nb keys
        sel = np.concatenate([np.arange(na[r]), La + np.arange(nb[r])])
        o1, l1 = at.attention_rows(q[r:r + 1], k[sel], v[sel], s)
        ou.append(o1[0])
        lu.append(l1[0])
    ou, lu = np.array(ou), np.array(lu)
    dev = lambda x: torch.from_numpy(np.where(np.isnan(x), 0.0, x).astype(np.float32)).cuda()
    o, l = L.lynx_attn_merge(dev(oa), dev(np.where(np.isfinite(la), la, -np.inf)), dev(ob),
                             dev(np.where(np.isfinite(lb), lb, -np.inf)))
    o, l = o.cpu().numpy(), l.cpu().numpy()
    empty = ~np.isfinite(lu)
    assert empty.sum() == 1 and np.all(o[empty] == 0.0) and np.all(np.isneginf(l[empty]))
    check_attention(o, l, np.nan_to_num(ou), lu, mask=~empty)
    # in place: the result may overwrite the first input
    a_o, a_l = dev(oa), dev(np.where(np.isfinite(la), la, -np.inf))
    L.lynx_attn_merge(a_o, a_l, dev(ob), dev(np.where(np.isfinite(lb), lb, -np.inf)), out=a_o, lse=a_l)
    assert np.array_equal(a_o.cpu().numpy(), o) and np.array_equal(a_l.cpu().numpy(), l)


@pytest.mark.parametrize("mode", ["anchor", "full"])
def test_verification_with_the_drafts_uncompressed_kv(cuda_device, mode):
    """T = 4 draft tokens, GQA 4:1, 2 KV heads: the context (1000 tokens, packed)
    is seen by every draft; the drafts' own K and V (BF16) causally."""
    Hkv, G, T, ctx = 2, 4, 4, 1000
    Hq = Hkv * G
    out = inputs.outlier_pairs(Hkv, 6)
    kb = inputs.kv_pages_np(Hkv, 1024, 61, out)            # [Hkv * 4 pages, 128, 256]
    vb = inputs.kv_pages_np(Hkv, 1024, 62, out)
    ka, kr, km = lo.encode_pages(kb, 100.0, EPS)
    va, vr, vm = lo.encode_pages(vb, 100.0, EPS)
    full = mode == "full"
    kd = lo.reconstruct(ka, kr if full else None, km, 100.0, EPS)
    vd = lo.reconstruct(va, vr if full else None, vm, 100.0, EPS)
    # the drafts' K and V: one BF16 page per KV head, first T tokens valid
    tk = inputs.kv_pages_np(Hkv, 256, 63, out)
    tv = inputs.kv_pages_np(Hkv, 256, 64, out)
    q = inputs.queries_np((1, T, Hq, 128), 65)
    cu = lambda x: torch.from_numpy(x).cuda()
    bf = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
    table = np.array([[[4 * h + p for p in range(4)] for h in range(Hkv)]], dtype=np.int32)
    o_c, l_c = L.lynx_decode_attn(bf(q), cu(ka), cu(kr) if full else None, cu(km), cu(va),
                                  cu(vr) if full else None, cu(vm), cu(table), cu(np.array([ctx], np.int32)),
                                  Hkv, causal=False)
    t_table = np.array([[[h] for h in range(Hkv)]], dtype=np.int32)
    o_t, l_t = L.lynx_decode_attn_bf16(bf(q), bf(tk), bf(tv), cu(t_table), cu(np.array([T], np.int32)), Hkv,
                                       causal=True)
    o, l = L.lynx_attn_merge(o_c, l_c, o_t, l_t)
    torch.cuda.synchronize()
    L.lynx_device_status()
    # oracle: each query row over the context keys then its visible drafts
    qf = lo.bf16_to_f32(q).astype(np.float64)[0]           # [T, Hq, 128]
    ro = np.zeros((1, T, Hq, 128))
    rl = np.zeros((1, T, Hq))
    for h in range(Hkv):
        k_seq = np.concatenate([at.pages_to_seq(kd[4 * h:4 * h + 4])[:ctx],
                                at.pages_to_seq(lo.bf16_to_f32(tk[h:h + 1]).astype(np.float64))[:T]])
        v_seq = np.concatenate([at.pages_to_seq(vd[4 * h:4 * h + 4])[:ctx],
                                at.pages_to_seq(lo.bf16_to_f32(tv[h:h + 1]).astype(np.float64))[:T]])
        rows = qf[:, h * G:(h + 1) * G, :].reshape(T * G, 128)
        nv = np.repeat(ctx + 1 + np.arange(T), G)
        oo, ll = at.attention_rows(rows, k_seq, v_seq, 1 / math.sqrt(128), nv)
        ro[0, :, h * G:(h + 1) * G] = oo.reshape(T, G, 128)
        rl[0, :, h * G:(h + 1) * G] = ll.reshape(T, G)
    check_attention(o.cpu().numpy(), l.cpu().numpy(), ro, rl)
