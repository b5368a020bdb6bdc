"""The Reindex selection in the form of the published reference code ([P1]
"DeepSeek V4.1 Flash 아키텍처 분석", §"공개 코드를 읽어 보니 남는 차이":
Indexer.forward scores every key, then masks the positions outside the
candidates) against scoring only inside the pool and against the oracle.  With
at least k visible positions in the pool both forms select the same positions."""
import numpy as np
import pytest
import torch

from fp4_compressed_sparse_gb300 import csa2
from gpu_util import build_r1, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp4_compressed_sparse_gb300 import build_lib
    build_lib.build()
    csa2.load()


@pytest.mark.parametrize("bs,nblk,k", [(8, 64, 64), (8, 300, 512), (4, 90, 100)])
def test_masked_full_scan_selects_like_the_pool(orc, bs, nblk, k):
    B, T, H_I = 3, 5000, 16
    c, oc, _, err = build_r1(orc, B, T, csa2.SWA_MXFP8, seed=91)
    g = torch.Generator().manual_seed(92)
    q_idx = torch.randn((B, H_I, 128), generator=g).to(torch.bfloat16).cuda()
    w = torch.rand((B, H_I), generator=g).cuda()
    Tv = T - 1
    q_pos = torch.full((B,), Tv, dtype=torch.int64, device="cuda")
    pool = torch.stack([torch.sort(torch.randperm((Tv + bs - 1) // bs, generator=g)[:nblk]).values
                        for _ in range(B)]).to(torch.int32)
    pool[2, -5:] = -1  # a shorter pool
    pool_d = pool.cuda()
    # pool-only scoring
    stride = nblk * bs
    ps = torch.empty((B, stride), device="cuda")
    aux = csa2.score_aux(B, stride)
    csa2.index_score(c, q_idx, w, q_pos, ps, pool=pool_d, pool_block_size=bs, err=err, aux=aux)
    idx_pool = torch.empty((B, k), dtype=torch.int32, device="cuda")
    csa2.topk(ps, 1, q_pos, k, idx_pool, csa2.topk_workspace(B, stride, k), pool=pool_d, pool_block_size=bs,
              err=err, aux=aux)
    # every position scored, then masked
    fs = torch.empty((B, c.capacity), device="cuda")
    csa2.index_score(c, q_idx, w, q_pos, fs, err=err)
    full = fs.clone()
    csa2.mask_to_pool(fs, 1, q_pos, pool_d, pool_block_size=bs)
    idx_mask = torch.empty((B, k), dtype=torch.int32, device="cuda")
    csa2.topk(fs, 1, q_pos, k, idx_mask, csa2.topk_workspace(B, c.capacity, k), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(idx_pool, idx_mask)
    for b in range(B):
        pl = pool[b].numpy()
        cnt = int((pl >= 0).sum())
        pos = orc.pool_positions(pl, cnt, Tv, bs)
        assert pos.shape[0] >= k
        ref, flags = orc.index_scores(oc[b], u16(q_idx[b]), w[b].cpu().numpy(), rows=pos)
        assert flags == 0
        assert idx_mask[b].tolist() == orc.topk(ref, k, positions=pos).tolist()
        # the mask: pool positions keep their scores bit for bit, the rest read -inf
        row, orig = fs[b, :Tv].cpu().numpy(), full[b, :Tv].cpu().numpy()
        inside = np.zeros(Tv, bool)
        inside[pos] = True
        assert np.array_equal(row[inside].view(np.uint32), orig[inside].view(np.uint32))
        assert np.array_equal(row[inside].view(np.uint32), ref.view(np.uint32))
        assert np.all(np.isneginf(row[~inside]))
