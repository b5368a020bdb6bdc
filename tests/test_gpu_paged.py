"""Paged KV ([P5] §3.5.1: global entries in fixed-size blocks named by a block
table; the window and the compression buffer are per-sequence state): a cache
whose pages are spread over a shuffled physical pool must give bit for bit the
records, scores, selections, attention outputs and prefill results of the
dense cache built from the same tokens (which the other parity tests check
against the oracle), and one sequence is also checked against the oracle here."""
import math

import numpy as np
import pytest
import torch

from fp4_compressed_sparse_gb300 import csa2
from fp4_compressed_sparse_gb300 import workloads as wl
from gpu_util import attn_close, cmp_rows, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp4_compressed_sparse_gb300 import build_lib
    build_lib.build()
    csa2.load()


def _shuffled_table(batch, max_pages, n_pages, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(n_pages, generator=g)[:batch * max_pages].to(torch.int32).view(batch, max_pages)


def _pair(batch, capacity, page, ratio=1, extra_pages=5, seed=0):
    max_pages = capacity // page
    n_pages = batch * max_pages + extra_pages
    paged = csa2.Cache(batch, capacity, ratio=ratio, page_entries=page, n_pages=n_pages,
                       block_table=_shuffled_table(batch, max_pages, n_pages, seed))
    return csa2.Cache(batch, capacity, ratio=ratio), paged


def _same_records(dense, paged, n):
    for name in ("lat_codes", "lat_scales", "rope_codes", "rope_scales"):
        assert torch.equal(dense.plane(name)[:, :n], paged.plane(name)[:, :n]), name
    for a, b in zip(dense.idx_entries(), paged.idx_entries()):
        assert torch.equal(a[:, :n], b[:, :n])
    assert torch.equal(dense.swa_codes, paged.swa_codes) and torch.equal(dense.n_tokens, paged.n_tokens)


@pytest.mark.parametrize("page", [128, 256])
def test_paged_decode_step_matches_dense(orc, page):
    B, cap, T, H, H_I, k = 3, 1024, 900, 64, 16, 64
    seed = 17
    caches = _pair(B, cap, page, seed=page)
    rope = csa2.rope_table(1e4, cap + 8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = 0
    for n in (300, 1, 599):
        kv = torch.stack([wl.token_rows(seed, wl.S_KV, b, t0, n, 576) for b in range(B)]).cuda()
        ik = torch.stack([wl.token_rows(seed, wl.S_IK, b, t0, n, 128) for b in range(B)]).cuda()
        for c in caches:
            csa2.kv_append(c, kv, ik, rope, err=err)
        t0 += n
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    dense, paged = caches
    _same_records(dense, paged, T)
    g = torch.Generator().manual_seed(seed + 1)
    q_idx = torch.randn((B, H_I, 128), generator=g).to(torch.bfloat16).cuda()
    w = torch.rand((B, H_I), generator=g).cuda()
    q = torch.randn((B, H, 576), generator=g).to(torch.bfloat16).cuda()
    q_pos = torch.tensor([T - 1, T - 60, 700], dtype=torch.int64, device="cuda")
    res = []
    for c in caches:
        scores = torch.full((B, cap), float("nan"), device="cuda")
        aux = csa2.score_aux(B, cap)
        csa2.index_score(c, q_idx, w, q_pos, scores, err=err, aux=aux)
        idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
        pool = torch.empty((B, 64), dtype=torch.int32, device="cuda")
        pcnt = torch.empty((B,), dtype=torch.int32, device="cuda")
        csa2.topk(scores, 1, q_pos, k, idx, csa2.topk_workspace(B, cap, k, 64), pool_out=pool, pool_count=pcnt,
                  err=err, aux=aux)
        # Reindex over that pool on the tensor cores (8-position blocks) and on CUDA cores (4)
        ps8 = torch.full((B, 64 * 8), float("nan"), device="cuda")  # slots of padded pool entries stay unwritten
        csa2.index_score(c, q_idx, w, q_pos, ps8, pool=pool, err=err)
        pool4 = torch.where(pool >= 0, pool * 2, -1).to(torch.int32)  # the first half of each 8-block
        ps4 = torch.full((B, 64 * 4), float("nan"), device="cuda")
        csa2.index_score(c, q_idx, w, q_pos, ps4, pool=pool4, pool_block_size=4, err=err)
        out = torch.empty((B, H, 512), device="cuda")
        lse = torch.empty((B, H), device="cuda")
        csa2.sparse_attn_decode(c, q, q_pos, idx, out, lse, csa2.attn_workspace(B, H, k), 1 / math.sqrt(576),
                                err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        res.append((scores, idx, pool, pcnt, ps8, ps4, out, lse))
    for (name, a, b) in zip(("scores", "idx", "pool", "pool count", "reindex scores", "4-block scores", "out",
                             "lse"), *res):
        if a.is_floating_point():
            a, b = a.nan_to_num(nan=7.0), b.nan_to_num(nan=7.0)  # slots past the visible ones stay unwritten
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), name
        else:
            assert torch.equal(a, b), name
    # one sequence against the oracle as well
    b = 1
    qp = int(q_pos[b])
    kc = orc.KeyCache(qp)
    orc.encode_keys(kc, 0, wl.token_rows(seed, wl.S_IK, b, 0, qp, 128).numpy())
    ref, flags = orc.index_scores(kc, u16(q_idx[b]), w[b].cpu().numpy(), n_vis=qp)
    assert flags == 0
    got = res[1][0][b, :qp].cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert res[1][1][b].tolist() == orc.topk(ref, k).tolist()


def test_paged_prefill_matches_dense():
    B, prior, Q, H_I, H, k, page, seed = 2, 500, 90, 64, 16, 32, 128, 23
    cap = 512  # 4 pages of 128 entries = 1,024 tokens at ratio 2
    caches = _pair(B, cap, page, ratio=2, seed=5)
    rope = csa2.rope_table(1e4, 2 * cap + 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = torch.Generator().manual_seed(seed)
    ba = torch.randn((2, 704), generator=g).cuda() * 0.5
    bb = torch.randn((2, 704), generator=g).cuda() * 0.5
    rows = [torch.stack(x).cuda() for x in zip(*[cmp_rows(seed, b, 0, prior) for b in range(B)])]
    for c in caches:
        csa2.kv_append(c, rope_cs=rope, cmp=rows + [ba, bb], err=err)
    seq = 1
    chunk = [r.cuda() for r in cmp_rows(seed, seq, prior, Q)]
    q_idx = torch.randn((Q, H_I, 128), generator=g).to(torch.bfloat16).cuda()
    w = torch.rand((Q, H_I), generator=g).cuda()
    q = torch.randn((Q, H, 576), generator=g).to(torch.bfloat16).cuda()
    outs = []
    for c in caches:
        idx = torch.empty((Q, k), dtype=torch.int32, device="cuda")
        out = torch.empty((Q, H, 512), device="cuda")
        lse = torch.empty((Q, H), device="cuda")
        csa2.prefill_chunk(c, seq, chunk + [ba, bb], rope, q_idx, w, q, k, 1 / math.sqrt(576), idx, out, lse,
                           csa2.prefill_workspace(Q, cap, H_I, H, k), err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append((idx, out, lse))
    _same_records(caches[0], caches[1], (prior + Q) // 2)
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int32) if a.is_floating_point() else a,
                          b.view(torch.int32) if b.is_floating_point() else b)


def test_page_id_outside_the_pool_is_reported():
    """A table entry naming a page beyond the pool: the append raises INDEX and
    writes nothing there; the score and the attention skip that page too."""
    B, cap, page = 1, 512, 128
    table = torch.tensor([[0, 1, 2, 9]], dtype=torch.int32)  # page 9 does not exist (4 pages)
    c = csa2.Cache(B, cap, page_entries=page, n_pages=4, block_table=table)
    rope = csa2.rope_table(1e4, cap + 8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv = torch.randn((B, 384, 576), device="cuda")
    ik = torch.randn((B, 384, 128), device="cuda")
    csa2.kv_append(c, kv, ik, rope, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0  # entries 0..383 live in pages 0..2; entry 384 on would be in page 9
    csa2.kv_append(c, torch.randn((B, 100, 576), device="cuda"), torch.randn((B, 100, 128), device="cuda"), rope,
                   err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & csa2.DEVERR_INDEX
    err.zero_()
    scores = torch.empty((B, cap), device="cuda")
    q_pos = torch.tensor([483], dtype=torch.int64, device="cuda")
    csa2.index_score(c, torch.randn((B, 4, 128), device="cuda").to(torch.bfloat16), torch.rand((B, 4),
                     device="cuda"), q_pos, scores, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & csa2.DEVERR_INDEX
