"""The V4 entry format ([P5] §2.3.4: KV entries in FP8 except the RoPE dims,
which stay BF16; here MXFP8 latent + bf16 RoPE, 656 B per main entry) through
the same kernels as the V4.1 FP4 record: append bytes bit-exact against the
oracle (ratio 1 and ratio 2), attention within 2e-3 of the oracle's fp64
attention over the dequantised entries (also with values beyond fp16 range),
a whole decode step and a prefill chunk."""
import math

import numpy as np
import pytest
import torch

from fp4_compressed_sparse_gb300 import csa2
from gpu_util import assert_cache_equal, attn_close, build_r1, build_r2, cmp_rows, u16

pytestmark = pytest.mark.gpu
FP8 = csa2.ENTRY_FP8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp4_compressed_sparse_gb300 import build_lib
    build_lib.build()
    csa2.load()


@pytest.mark.parametrize("swa_dtype", [csa2.SWA_BF16, csa2.SWA_MXFP8])
def test_v4_append_r1_bitexact(orc, swa_dtype):
    c, oc, _, err = build_r1(orc, 2, 301, swa_dtype, seed=101, chunks=[150, 1, 150], entry_format=FP8)
    assert int(err.item()) == 0
    assert c.entry_bytes() == 528 + 128 + 68
    assert_cache_equal(c, oc, 301)


def test_v4_append_r2_bitexact(orc):
    c, oc, _, err, _, _, _ = build_r2(orc, 2, 90, csa2.SWA_MXFP8, seed=102, chunks=[31, 1, 58], entry_format=FP8)
    assert int(err.item()) == 0
    assert_cache_equal(c, oc, 45)


@pytest.mark.parametrize("B,T,H,k,kv_scale,use_sink", [
    (3, 700, 64, 64, 1.0, False),
    (32, 300, 64, 128, 1.0, True),        # 4 CTAs per row
    (2, 500, 64, 256, 2.0 ** 18, False),  # latent and RoPE values beyond fp16: a power-of-two scale per entry
    (1, 90, 16, 64, 1.0, True),           # window shorter than 128
    (2, 600, 64, 599, 1.0, False),        # every visible entry selected: the dense (HCA-style) layer
])
def test_v4_sparse_attn(orc, B, T, H, k, kv_scale, use_sink):
    c, oc, _, err = build_r1(orc, B, T, csa2.SWA_MXFP8, seed=103 + B, kv_scale=kv_scale, entry_format=FP8)
    g = torch.Generator().manual_seed(104)
    q = torch.randn((B, H, 576), generator=g)
    if kv_scale != 1.0:
        q = q / kv_scale
    q = q.to(torch.bfloat16)
    Tv = T - 1
    idx = torch.full((B, k), -1, dtype=torch.int32)
    for b in range(B):
        n = min(k, Tv) - (b % 2)
        idx[b, :n] = torch.sort(torch.randperm(Tv, generator=g)[:n]).values.to(torch.int32)
    sink = (torch.randn(H, generator=g) * 2).float() if use_sink else None
    q_pos = torch.full((B,), Tv, dtype=torch.int64, device="cuda")
    out = torch.empty((B, H, 512), device="cuda")
    lse = torch.empty((B, H), device="cuda")
    scale = 1 / math.sqrt(576)
    csa2.sparse_attn_decode(c, q.cuda(), q_pos, idx.cuda(), out, lse, csa2.attn_workspace(B, H, k), scale,
                            sink=sink.cuda() if sink is not None else None, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for b in range(B):
        ro, rl = orc.sparse_attn(oc[b], u16(q[b]), idx[b].numpy(), Tv, scale,
                                 sink.numpy() if sink is not None else None)
        attn_close(out[b].cpu().numpy(), lse[b].cpu().numpy(), ro, rl)


def test_v4_decode_step(orc):
    B, T, H, H_I, k = 2, 3000, 64, 16, 128
    c, oc, _, err = build_r1(orc, B, T, csa2.SWA_MXFP8, seed=105, entry_format=FP8)
    g = torch.Generator().manual_seed(106)
    q_idx = torch.randn((B, H_I, 128), generator=g).to(torch.bfloat16)
    w = torch.rand((B, H_I), generator=g)
    q = torch.randn((B, H, 576), generator=g).to(torch.bfloat16)
    q_pos = torch.full((B,), T - 1, dtype=torch.int64, device="cuda")
    scores = torch.empty((B, c.capacity), device="cuda")
    aux = csa2.score_aux(B, c.capacity)
    csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores, err=err, aux=aux)
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    csa2.topk(scores, 1, q_pos, k, idx, csa2.topk_workspace(B, c.capacity, k), err=err, aux=aux)
    out = torch.empty((B, H, 512), device="cuda")
    lse = torch.empty((B, H), device="cuda")
    scale = 1 / math.sqrt(576)
    csa2.sparse_attn_decode(c, q.cuda(), q_pos, idx, out, lse, csa2.attn_workspace(B, H, k), scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for b in range(B):
        r_idx, _, _, ro, rl, r_scores = orc.full_layer(oc[b], u16(q_idx[b]), w[b].numpy(), u16(q[b]), T - 1, k, scale)
        assert np.array_equal(scores[b, :T - 1].cpu().numpy().view(np.uint32), r_scores.view(np.uint32))
        assert idx[b].tolist() == r_idx.tolist()
        attn_close(out[b].cpu().numpy(), lse[b].cpu().numpy(), ro, rl)


def test_v4_prefill_chunk(orc):
    prior, Q, H_I, H, k = 200, 30, 4, 16, 32
    c, oc, rope, err, (ba, bb), _, _ = build_r2(orc, 1, prior, csa2.SWA_MXFP8, seed=107, cap=(prior + Q) // 2 + 8,
                                               entry_format=FP8)
    rows = cmp_rows(107, 0, prior, Q)
    g = torch.Generator().manual_seed(108)
    q_idx = torch.randn((Q, H_I, 128), generator=g).to(torch.bfloat16)
    w = torch.rand((Q, H_I), generator=g)
    q = torch.randn((Q, H, 576), generator=g).to(torch.bfloat16)
    idx = torch.empty((Q, k), dtype=torch.int32, device="cuda")
    out = torch.empty((Q, H, 512), device="cuda")
    lse = torch.empty((Q, H), device="cuda")
    scale = 1 / math.sqrt(576)
    csa2.prefill_chunk(c, 0, [r.cuda() for r in rows] + [ba.cuda(), bb.cuda()], rope, q_idx.cuda(), w.cuda(),
                       q.cuda(), k, scale, idx, out, lse, csa2.prefill_workspace(Q, c.capacity, H_I, H, k), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o = oc[0]
    prior_ring = {t: (o.swa_codes[t % 128].copy(), o.swa_scales[t % 128].copy())
                  for t in range(max(0, prior - 128), prior)}
    orc.append_r2(o, *[r.numpy() for r in rows], ba.numpy(), bb.numpy(), 1e4)
    assert_cache_equal(c, [o], (prior + Q) // 2, check_swa=False)
    for i in (0, 13, Q - 1):
        t = prior + i
        sc, flags = orc.index_scores(o, u16(q_idx[i]), w[i].numpy(), n_vis=t // 2)
        r_idx = orc.topk(sc, k)
        assert idx[i].tolist() == r_idx.tolist()
        toks = list(range(max(0, t - 127), t + 1))
        recs = [(orc.encode_swa(rows[0][x - prior, :576].numpy(), orc.rope_cs(1e4, x), csa2.SWA_MXFP8)
                 if x >= prior else prior_ring[x]) for x in toks]
        ro, rl = orc.sparse_attn(o, u16(q[i]), r_idx, t, scale, swa_codes=np.array([r[0] for r in recs]),
                                 swa_scales=np.array([r[1] for r in recs]))
        attn_close(out[i].cpu().numpy(), lse[i].cpu().numpy(), ro, rl)
