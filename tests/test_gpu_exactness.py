"""GPU parity of the index score at the edge of its exactness bound, and on the
CUDA-core path (pool blocks of other sizes than 8).

The block-scaled dot of an MXFP4 query head and key is an integer multiple of
its smallest block's unit, below 2^(15 + span) with span = max - min of the
pair's block exponents e_q,j + e_k,j ([P5] §2.3.4 puts the indexer QK product
in FP4; the bound is arithmetic on the E2M1 grid: a 32-wide block sum of
doubled codes is below 2^13).  At span 9 it still fits the fp32 significand, so
the score must equal the oracle's exact dot rounded once; beyond it the library
raises CSA2_DEVERR_INEXACT.
"""
import numpy as np
import pytest
import torch

from fp4_compressed_sparse_gb300 import csa2
from gpu_util import u16

pytestmark = pytest.mark.gpu

GRID = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float32)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp4_compressed_sparse_gb300 import build_lib
    build_lib.build()
    csa2.load()


def _mx_rows(rng, n, exps, extreme):
    """n rows of 128 values on the E2M1 grid times 2^exps[j] in block j, each block's
    first value +-6 * 2^exps[j] (so its MXFP4 exponent is exps[j], and quantisation is
    exact).  exps[j] = None leaves block j all zero.  `extreme` pushes block 3 to
    its largest integer sum (every value +6) and blocks 0..2 to the smallest."""
    x = np.zeros((n, 128), np.float32)
    for j, e in enumerate(exps):
        if e is None:
            continue
        if extreme and j == 3:
            blk = np.full((n, 32), 6.0, np.float32)
        elif extreme:
            blk = np.zeros((n, 32), np.float32)
            blk[:, 0] = 6.0
            blk[:, 1] = 0.5 * rng.choice([-1.0, 1.0], size=n)
        else:
            blk = rng.choice(GRID, size=(n, 32)) * rng.choice([-1.0, 1.0], size=(n, 32))
            blk[:, 0] = 6.0 * rng.choice([-1.0, 1.0], size=n)
        x[:, 32 * j:32 * j + 32] = blk * np.float32(2.0 ** e)
    return x


def _run(orc, key_exps, q_exps, extreme, mode, seed):
    """Keys with the given block exponents in a ratio-1 cache; queries with theirs;
    scores through FULL (tensor cores), POOL with 8-position blocks (tensor cores,
    gathered) or POOL with 4-position blocks (CUDA cores).  Returns (err word,
    GPU scores of the visible slots, oracle scores, oracle flags)."""
    rng = np.random.default_rng(seed)
    B, T, H = 1, 600, 8
    cap = T + 8
    c = csa2.Cache(B, cap, ratio=1)
    rope = csa2.rope_table(1e4, cap + 8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ik = _mx_rows(rng, T, key_exps, extreme)
    kv = rng.standard_normal((T, 576)).astype(np.float32)
    csa2.kv_append(c, torch.from_numpy(kv)[None].cuda(), torch.from_numpy(ik)[None].cuda(), rope, err=err)
    kc = orc.KeyCache(T)
    orc.encode_keys(kc, 0, ik)
    q = _mx_rows(rng, H, q_exps, extreme)
    q_idx = torch.from_numpy(q).to(torch.bfloat16)[None]
    assert torch.equal(q_idx[0].float(), torch.from_numpy(q))  # grid values are exact in bf16
    w = torch.from_numpy(rng.random((B, H)).astype(np.float32))
    q_pos = torch.full((B,), T - 1, dtype=torch.int64, device="cuda")
    Tv = T - 1
    if mode == "full":
        scores = torch.empty((B, cap), device="cuda")
        csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores, err=err)
        torch.cuda.synchronize()
        got = scores[0, :Tv].cpu().numpy()
        ref, flags = orc.index_scores(kc, u16(q_idx[0]), w[0].numpy(), n_vis=Tv)
        return int(err.item()), got, ref, flags
    bs = 8 if mode == "pool8" else 4
    nb = (Tv + bs - 1) // bs
    pids = np.sort(rng.choice(nb, size=min(40, nb), replace=False)).astype(np.int32)
    pool = torch.from_numpy(pids)[None].cuda()
    stride = len(pids) * bs
    scores = torch.empty((B, stride), device="cuda")
    csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores, pool=pool, pool_block_size=bs, err=err)
    torch.cuda.synchronize()
    pos = orc.pool_positions(pids, len(pids), Tv, bs)
    slots = np.array([list(pids).index(p // bs) * bs + p % bs for p in pos])
    got = scores[0].cpu().numpy()[slots]
    ref, flags = orc.index_scores(kc, u16(q_idx[0]), w[0].numpy(), rows=pos)
    return int(err.item()), got, ref, flags


@pytest.mark.parametrize("mode", ["full", "pool8", "pool4"])
@pytest.mark.parametrize("extreme", [False, True])
def test_span_nine_is_exact(orc, mode, extreme):
    """Key blocks at exponents (0, 0, 0, 9) against query blocks at (0, 0, 0, 0):
    every pair spans exactly 9 binades.  With `extreme` the block-3 sum is the
    largest possible (32 x 12 x 12 doubled codes) and blocks 0..2 add a few units:
    a 22-bit integer, still exact in fp32.  Scores bit-exact, no INEXACT bit."""
    err, got, ref, flags = _run(orc, (0, 0, 0, 9), (0, 0, 0, 0), extreme, mode, seed=5)
    assert flags == 0
    assert err & csa2.DEVERR_INEXACT == 0
    assert err == 0
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"{np.sum(got != ref)} scores differ"


@pytest.mark.parametrize("mode", ["full", "pool8", "pool4"])
@pytest.mark.parametrize("key_exps,q_exps", [
    ((0, 0, 0, 12), (0, 0, 0, 0)),     # the key alone spans 12
    ((0, 5, 0, 0), (-5, 0, 1, 1)),     # each spans 5-6; the pair (e_q + e_k) spans 10
])
def test_span_beyond_nine_raises_inexact(orc, mode, key_exps, q_exps):
    err, got, ref, flags = _run(orc, key_exps, q_exps, True, mode, seed=6)
    assert err & csa2.DEVERR_INEXACT


@pytest.mark.parametrize("mode", ["full", "pool8", "pool4"])
def test_zero_block_takes_no_part(orc, mode):
    """A key block that is all zero (scale code 0) against query blocks spanning
    9: the zero block contributes nothing, the bound holds, scores are exact."""
    err, got, ref, flags = _run(orc, (None, 0, 0, 0), (0, 0, 9, 0), False, mode, seed=7)
    assert flags == 0 and err == 0
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("bs", [4, 16])
def test_pool_other_block_sizes_against_oracle(orc, bs):
    """Reindex scoring with pool blocks of 4 and 16 positions (the CUDA-core score
    path) and the top-k inside the pool, with and without the score sideband,
    against the oracle over the pool's visible positions."""
    from gpu_util import build_r1
    B, T, H_I, k = 2, 2500, 16, 64
    c, oc, _, err = build_r1(orc, B, T, csa2.SWA_MXFP8, seed=81)
    g = torch.Generator().manual_seed(82)
    q_idx = torch.randn((B, H_I, 128), generator=g).to(torch.bfloat16)
    w = torch.rand((B, H_I), generator=g)
    Tv = T - 1
    q_pos = torch.full((B,), Tv, dtype=torch.int64, device="cuda")
    nblk = 50
    pools = [torch.sort(torch.randperm((Tv + bs - 1) // bs, generator=g)[:nblk]).values.to(torch.int32)
             for _ in range(B)]
    pool = torch.stack(pools)
    pool[1, -4:] = -1  # a short pool
    stride = nblk * bs
    scores = torch.empty((B, stride), device="cuda")
    aux = csa2.score_aux(B, stride)
    csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores, pool=pool.cuda(), pool_block_size=bs, err=err,
                     aux=aux)
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    idx2 = torch.empty_like(idx)
    ws = csa2.topk_workspace(B, stride, k)
    csa2.topk(scores, 1, q_pos, k, idx, ws, pool=pool.cuda(), pool_block_size=bs, err=err, aux=aux)
    csa2.topk(scores, 1, q_pos, k, idx2, ws, pool=pool.cuda(), pool_block_size=bs, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(idx, idx2)
    for b in range(B):
        pl = pool[b].numpy()
        cnt = int((pl >= 0).sum())
        pos = orc.pool_positions(pl, cnt, Tv, bs)
        ref, flags = orc.index_scores(oc[b], u16(q_idx[b]), w[b].numpy(), rows=pos)
        assert flags == 0
        slots = np.array([list(pl[:cnt]).index(p // bs) * bs + p % bs for p in pos])
        got = scores[b].cpu().numpy()[slots]
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"row {b}"
        assert idx[b].tolist() == orc.topk(ref, k, positions=pos).tolist(), f"row {b} top-k"
