"""GPU parity: libcsa2 (through the C ABI) against the CPU oracle on the same
seeded inputs.  Codes, scales, scores, indices and pool ids bit-exact;
attention within 2e-3 normwise per head (and lse within 2e-3)."""
import math

import numpy as np
import pytest
import torch

from fp4_compressed_sparse_gb300 import csa2
from fp4_compressed_sparse_gb300 import workloads as wl

from gpu_util import assert_cache_equal, attn_close, build_r1, build_r2, cmp_rows, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp4_compressed_sparse_gb300 import build_lib
    build_lib.build()
    csa2.load()


# ------------------------------------------------------------------ append
@pytest.mark.parametrize("swa_dtype", [csa2.SWA_BF16, csa2.SWA_MXFP8])
@pytest.mark.parametrize("in_bf16", [False, True])
def test_append_r1_bitexact(orc, swa_dtype, in_bf16):
    c, oc, _, err = build_r1(orc, 2, 201, swa_dtype, seed=11, chunks=[130, 1, 70], in_bf16=in_bf16)
    assert int(err.item()) == 0
    assert c.n_tokens.tolist() == [201, 201]
    assert_cache_equal(c, oc, 201)


def test_append_r2_bitexact(orc):
    c, oc, _, err, _, gdbg, odbg = build_r2(orc, 2, 100, csa2.SWA_MXFP8, seed=12, chunks=[7, 30, 1, 62],
                                            dbg=True)
    assert int(err.item()) == 0
    assert c.n_tokens.tolist() == [100, 100]
    # compressed fp32 rows (before RoPE): both sides compute in fp64 and round once
    for b in range(2):
        got = []
        t0 = 0
        for d, n in zip(gdbg, [7, 30, 1, 62]):
            n_emit = (t0 + n) // 2 - t0 // 2
            got += list(d[b, :n_emit].cpu().numpy())
            t0 += n
        ref = np.array(odbg[b])
        got = np.array(got)
        assert got.shape == ref.shape == (50, 704)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert_cache_equal(c, oc, 50)


def test_append_capacity_error():
    c = csa2.Cache(1, 4, ratio=1)
    rope = csa2.rope_table(1e4, 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv = torch.randn(1, 5, 576, device="cuda")
    ik = torch.randn(1, 5, 128, device="cuda")
    csa2.kv_append(c, kv, ik, rope, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & csa2.DEVERR_CAPACITY
    assert c.n_tokens.item() == 0 and not c.lat_codes.any()


# ------------------------------------------------------------------ scores / top-k / pool
def _decode_inputs(B, H_I, H, seed, step=0):
    g = torch.Generator().manual_seed(seed)
    q_idx = torch.randn((B, H_I, 128), generator=g).to(torch.bfloat16)
    w = torch.rand((B, H_I), generator=g)
    q = torch.randn((B, H, 576), generator=g).to(torch.bfloat16)
    return q_idx, w, q


@pytest.mark.parametrize("H_I", [4, 20, 64, 128])
def test_index_score_full_and_topk_bitexact(orc, H_I):
    B, T = 2, 1500
    c, oc, _, err = build_r1(orc, B, T, csa2.SWA_MXFP8, seed=21)
    q_idx, w, _ = _decode_inputs(B, H_I, 16, seed=22)
    q_pos = torch.full((B,), T - 1, dtype=torch.int64, device="cuda")
    scores = torch.full((B, c.capacity), float("nan"), device="cuda")
    csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores, err=err)
    k = 100
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    pool = torch.empty((B, 32), dtype=torch.int32, device="cuda")
    pcount = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = csa2.topk_workspace(B, c.capacity, k, 32)
    csa2.topk(scores, 1, q_pos, k, idx, ws, pool_out=pool, pool_count=pcount, err=err)
    # the same selection from the sideband the score kernel leaves
    aux = csa2.score_aux(B, c.capacity)
    scores2 = torch.full_like(scores, float("nan"))
    csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores2, err=err, aux=aux)
    idx2, pool2, pcount2 = torch.empty_like(idx), torch.empty_like(pool), torch.empty_like(pcount)
    csa2.topk(scores2, 1, q_pos, k, idx2, ws, pool_out=pool2, pool_count=pcount2, err=err, aux=aux)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(idx, idx2) and torch.equal(pool, pool2) and torch.equal(pcount, pcount2)
    Tv = T - 1
    for b in range(B):
        ref, flags = orc.index_scores(oc[b], u16(q_idx[b]), w[b].numpy(), n_vis=Tv)
        assert flags == 0
        got = scores[b, :Tv].cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), \
            f"{np.sum(got != ref)} scores differ"
        assert idx[b].tolist() == orc.topk(ref, k).tolist()
        pids, cnt = orc.pool(ref, Tv, 8, 32)
        assert pcount[b].item() == cnt and pool[b].tolist() == pids.tolist()


def test_index_score_many_short_rows_bitexact(orc):
    """More rows than SMs over a short context (a CTA's item range spans several
    rows, each with its own query record in the scan's operand slots), rows seeing
    different numbers of positions."""
    B, T, H_I = 200, 300, 64
    c, oc, _, err = build_r1(orc, B, T, csa2.SWA_MXFP8, seed=23)
    q_idx, w, _ = _decode_inputs(B, H_I, 16, seed=24)
    pos = [T - 1 - (b % 50) * 3 for b in range(B)]
    q_pos = torch.tensor(pos, dtype=torch.int64, device="cuda")
    scores = torch.full((B, c.capacity), float("nan"), device="cuda")
    csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for b in list(range(0, B, 7)) + [B - 1]:
        ref, flags = orc.index_scores(oc[b], u16(q_idx[b]), w[b].numpy(), n_vis=pos[b])
        assert flags == 0
        got = scores[b, :pos[b]].cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"row {b}: {np.sum(got != ref)} scores differ"


def test_index_score_block_scale_spread(orc):
    """Keys whose four 32-dim blocks differ in magnitude by up to 2^6 (and queries by
    up to 2^2): the block-scaled tensor-core dot must still equal the exact dot."""
    from gpu_util import build_r1  # noqa: F401
    B, T, H_I = 1, 700, 16
    cap = T + 8
    c = csa2.Cache(B, cap, ratio=1)
    rope = csa2.rope_table(1e4, cap + 8)
    oc = orc.Cache(cap)
    g = torch.Generator().manual_seed(71)
    kv = torch.randn((T, 576), generator=g)
    ik = torch.randn((T, 128), generator=g)
    fac = torch.tensor([2.0 ** -3, 1.0, 2.0 ** 3, 0.5]).repeat_interleave(32)
    ik = ik * fac
    csa2.kv_append(c, kv[None].cuda(), ik[None].cuda(), rope)
    orc.append_r1(oc, kv.numpy(), ik.numpy(), 1e4)
    q_idx = (torch.randn((B, H_I, 128), generator=g) *
             torch.tensor([1.0, 2.0, 0.5, 4.0]).repeat_interleave(32)).to(torch.bfloat16)
    w = torch.rand((B, H_I), generator=g)
    q_pos = torch.full((B,), T - 1, dtype=torch.int64, device="cuda")
    scores = torch.empty((B, cap), device="cuda")
    csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores)
    torch.cuda.synchronize()
    ref, flags = orc.index_scores(oc, u16(q_idx[0]), w[0].numpy(), n_vis=T - 1)
    assert flags == 0
    got = scores[0, :T - 1].cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_topk_ties_zero_weight_and_short_context(orc):
    B, T = 1, 300
    c, oc, _, err = build_r1(orc, B, T, csa2.SWA_MXFP8, seed=23)
    q_idx, _, _ = _decode_inputs(B, 4, 16, seed=24)
    w = torch.zeros((B, 4))
    scores = torch.empty((B, c.capacity), device="cuda")
    for qp, k in ((T - 1, 64), (40, 64), (0, 16), (1, 16)):
        q_pos = torch.full((B,), qp, dtype=torch.int64, device="cuda")
        csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores, err=err)
        idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
        ws = csa2.topk_workspace(B, c.capacity, k)
        csa2.topk(scores, 1, q_pos, k, idx, ws, err=err)
        torch.cuda.synchronize()
        want = list(range(min(qp, k))) + [-1] * (k - min(qp, k))  # all-zero scores: lowest positions
        assert idx[0].tolist() == want


def test_reindex_pool_bitexact(orc):
    B, T, H_I, nblk = 2, 3000, 8, 40
    c, oc, _, err = build_r1(orc, B, T, csa2.SWA_MXFP8, seed=31)
    q_idx, w, _ = _decode_inputs(B, H_I, 16, seed=32)
    q_pos = torch.full((B,), T - 1, dtype=torch.int64, device="cuda")
    g = torch.Generator().manual_seed(33)
    pools = []
    for b in range(B):
        p = torch.sort(torch.randperm((T - 1) // 8 + 1, generator=g)[:nblk]).values.to(torch.int32)
        pools.append(p)
    pool = torch.stack(pools)
    pool[1, -3:] = -1  # a short pool (padded)
    stride = nblk * 8
    scores = torch.empty((B, stride), device="cuda")
    csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores, pool=pool.cuda(), err=err)
    k = 64
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    ws = csa2.topk_workspace(B, stride, k)
    csa2.topk(scores, 1, q_pos, k, idx, ws, pool=pool.cuda(), err=err)
    aux = csa2.score_aux(B, stride)
    scores2 = torch.empty_like(scores)
    csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores2, pool=pool.cuda(), err=err, aux=aux)
    idx2 = torch.empty_like(idx)
    csa2.topk(scores2, 1, q_pos, k, idx2, ws, pool=pool.cuda(), err=err, aux=aux)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(idx, idx2)
    for b in range(B):
        pl = pool[b].numpy()
        cnt = int((pl >= 0).sum())
        pos = orc.pool_positions(pl, cnt, T - 1)
        ref, flags = orc.index_scores(oc[b], u16(q_idx[b]), w[b].numpy(), rows=pos)
        assert flags == 0
        # slot j of the score row is position pool[j//8]*8 + j%8
        slots = np.array([list(pl[:cnt]).index(p // 8) * 8 + p % 8 for p in pos])
        got = scores[b].cpu().numpy()[slots]
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        assert idx[b].tolist() == orc.topk(ref, k, positions=pos).tolist()


@pytest.mark.parametrize("levels,T,k,nblk", [
    (4, 30000, 512, 2048),     # four distinct values: the threshold bin holds ~7,500 scores
    (1, 9000, 100, 64),        # one value: every score ties, lowest positions win
    (0, 70000, 2048, 2048),    # continuous scores, k and pool at their maxima
    (3, 4000, 2048, 2048),     # fewer visible entries than k: everything is chosen
    (2, 5001, 64, 100),        # an odd row stride (unaligned rows take the scalar pass)
])
def test_topk_crowded_bins_against_oracle(orc, levels, T, k, nblk):
    """Scores written directly (not from the indexer): heavy ties and crowded
    histogram bins, both signs and -0/+0, FULL rows with the pool build."""
    B = 2
    g = torch.Generator().manual_seed(1000 + levels)
    stride = T + 40
    if levels:
        vals = torch.tensor([-0.0, 0.0, 1.5, -2.25, 1.5 + 2 ** -20][:levels + 1])
        sc = vals[torch.randint(0, len(vals), (B, stride), generator=g)]
    else:
        sc = torch.randn((B, stride), generator=g) * 3
    sc = sc.float().contiguous()
    q_pos = torch.tensor([T, T // 2 + 3], dtype=torch.int64)
    if T == 4000:
        q_pos = torch.tensor([1500, 7], dtype=torch.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    pool = torch.empty((B, nblk), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = csa2.topk_workspace(B, stride, k, nblk)
    csa2.topk(sc.cuda(), 1, q_pos.cuda(), k, idx, ws, pool_out=pool, pool_count=cnt, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for b in range(B):
        Tv = int(q_pos[b])
        row = sc[b, :Tv].numpy()
        assert idx[b].tolist() == orc.topk(row, k).tolist()
        pids, n = orc.pool(row, Tv, 8, nblk)
        assert cnt[b].item() == n and pool[b].tolist() == pids.tolist()


@pytest.mark.parametrize("levels", [0, 2, 4])
def test_topk_many_rows_against_oracle(orc, levels):
    """More (row, problem) pairs than one wave of four-CTA clusters holds, so the
    selector runs one CTA per (row, problem): heavy ties and crowded bins, both
    signs and -0/+0, rows of every length down to none, and the pool build; every
    row against the oracle."""
    B, T, k, nblk = 96, 20000, 512, 2048
    g = torch.Generator().manual_seed(2000 + levels)
    stride = T + 40
    if levels:
        vals = torch.tensor([-0.0, 0.0, 1.5, -2.25, 1.5 + 2 ** -20][:levels + 1])
        sc = vals[torch.randint(0, len(vals), (B, stride), generator=g)]
    else:
        sc = torch.randn((B, stride), generator=g) * 3
    sc = sc.float().contiguous()
    lens = [max(0, T - 211 * b) for b in range(B)]
    q_pos = torch.tensor(lens, dtype=torch.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    pool = torch.empty((B, nblk), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = csa2.topk_workspace(B, stride, k, nblk)
    csa2.topk(sc.cuda(), 1, q_pos.cuda(), k, idx, ws, pool_out=pool, pool_count=cnt, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    idx, pool, cnt = idx.cpu(), pool.cpu(), cnt.cpu()
    for b in range(B):
        row = sc[b, :lens[b]].numpy()
        assert idx[b].tolist() == orc.topk(row, k).tolist(), f"row {b} (T {lens[b]})"
        pids, n = orc.pool(row, lens[b], 8, nblk)
        assert cnt[b].item() == n and pool[b].tolist() == pids.tolist(), f"row {b} pool"


def test_topk_many_pool_rows_against_oracle(orc):
    """POOL rows (a Reindex layer's candidate pools), more of them than one wave of
    four-CTA clusters holds: one CTA per row, against the oracle over the pool's
    visible positions."""
    B, T, k, nblk = 100, 6000, 128, 96
    g = torch.Generator().manual_seed(77)
    pools = []
    for b in range(B):
        p = torch.sort(torch.randperm((T - 1) // 8 + 1, generator=g)[:nblk]).values.to(torch.int32)
        if b % 3 == 1 and b % 17:
            p[-(b % 17):] = -1  # padded pools
        pools.append(p)
    pool = torch.stack(pools)
    stride = nblk * 8
    vals = torch.tensor([0.5, 0.75, -1.0, 2.0])
    sc = torch.where(torch.rand((B, stride), generator=g) < 0.5, vals[torch.randint(0, 4, (B, stride), generator=g)],
                     torch.randn((B, stride), generator=g)).float().contiguous()
    q_pos = torch.tensor([T - 1 - 13 * b for b in range(B)], dtype=torch.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    ws = csa2.topk_workspace(B, stride, k)
    csa2.topk(sc.cuda(), 1, q_pos.cuda(), k, idx, ws, pool=pool.cuda(), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    idx = idx.cpu()
    for b in range(B):
        pl = pool[b].numpy()
        cnt = int((pl >= 0).sum())
        Tv = int(q_pos[b])
        pos = orc.pool_positions(pl, cnt, Tv)
        slots = np.array([list(pl[:cnt]).index(p // 8) * 8 + p % 8 for p in pos], dtype=np.int64)
        ref = sc[b].numpy()[slots] if len(slots) else np.zeros(0, np.float32)
        assert idx[b].tolist() == orc.topk(ref, k, positions=pos).tolist(), f"row {b}"


def test_topk_nan_score_is_reported(orc):
    sc = torch.randn((1, 5000))
    sc[0, 123] = float("nan")
    q_pos = torch.tensor([5000], dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.empty((1, 64), dtype=torch.int32, device="cuda")
    csa2.topk(sc.cuda(), 1, q_pos, 64, idx, csa2.topk_workspace(1, 5000, 64), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & csa2.DEVERR_NAN
    assert 123 not in idx[0].tolist()


@pytest.mark.parametrize("reps,k", [
    (1, 512),   # 4 rows: 4-CTA clusters
    (25, 512),  # 100 rows: one CTA per row
    (1, 4),     # small k: the threshold bin sits among the finite or the +inf scores
    (1, 5),
])
def test_topk_infinite_scores(orc, reps, k):
    """Rows whose k-th score is -inf (fewer finite scores than k: the threshold
    bin is the one that holds -inf), rows whose top is +inf (more +inf scores
    than k: the bin that holds +inf), and infinities scattered in a normal row,
    for the top-k and a 64-block pool, against the oracle."""
    T, nblk = 6000, 64
    rng = np.random.default_rng(77)
    sc = rng.standard_normal((4, T)).astype(np.float32)
    sc[0, 300:] = -np.inf
    sc[1, rng.choice(T, 10, replace=False)] = np.inf
    sc[1, rng.choice(T, 5, replace=False)] = -np.inf
    sc[2, :] = -np.inf
    sc[3, rng.choice(T, 600, replace=False)] = np.inf
    sc = np.ascontiguousarray(np.tile(sc, (reps, 1)))
    B = sc.shape[0]
    q_pos = torch.full((B,), T, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    pool = torch.empty((B, nblk), dtype=torch.int32, device="cuda")
    pcnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    csa2.topk(torch.from_numpy(sc).cuda(), 1, q_pos, k, idx, csa2.topk_workspace(B, T, k, nblk),
              pool_out=pool, pool_count=pcnt, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for b in range(B):
        assert idx[b].tolist() == orc.topk(sc[b], k).tolist(), f"row {b}: top-k"
        pids, cnt = orc.pool(sc[b], T, 8, nblk)
        assert int(pcnt[b].item()) == cnt and pool[b].tolist() == pids.tolist(), f"row {b}: pool"


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("B,T,H,k,swa_dtype,use_sink", [
    (3, 700, 64, 64, csa2.SWA_MXFP8, False),   # 4 segments, one per CTA; 16-head blocks
    (3, 700, 64, 64, csa2.SWA_BF16, True),
    (32, 200, 64, 48, csa2.SWA_MXFP8, True),   # 4 CTAs per row, 64 heads each
    (80, 200, 64, 48, csa2.SWA_BF16, False),   # one CTA per row computes all 4 segments
    (1, 90, 32, 128, csa2.SWA_MXFP8, False),   # window shorter than 128, idx padded with -1
    (3, 1500, 128, 1024, csa2.SWA_BF16, True), # 8 head blocks of 16, 9 chunks per segment
    (2, 300, 48, 200, csa2.SWA_MXFP8, False),  # 48 heads in blocks of 16
])
def test_sparse_attn_decode(orc, B, T, H, k, swa_dtype, use_sink):
    c, oc, _, err = build_r1(orc, B, T, swa_dtype, seed=41 + B)
    _, _, q = _decode_inputs(B, 4, H, seed=42)
    g = torch.Generator().manual_seed(43)
    Tv = T - 1
    idx = torch.full((B, k), -1, dtype=torch.int32)
    for b in range(B):
        n = min(k, Tv) - (b % 3)
        idx[b, :n] = torch.sort(torch.randperm(Tv, generator=g)[:n]).values.to(torch.int32)
    sink = (torch.randn(H, generator=g) * 2).float() if use_sink else None
    q_pos = torch.full((B,), T - 1, dtype=torch.int64, device="cuda")
    out = torch.empty((B, H, 512), device="cuda")
    lse = torch.empty((B, H), device="cuda")
    ws = csa2.attn_workspace(B, H, k)
    scale = 1 / math.sqrt(576)
    csa2.sparse_attn_decode(c, q.cuda(), q_pos, idx.cuda(), out, lse, ws, scale,
                            sink=sink.cuda() if sink is not None else None, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for b in range(B):
        ro, rl = orc.sparse_attn(oc[b], u16(q[b]), idx[b].numpy(), T - 1, scale,
                                 sink.numpy() if sink is not None else None)
        attn_close(out[b].cpu().numpy(), lse[b].cpu().numpy(), ro, rl)
    # Reuse identity: same query, same list, same cache -> identical bits
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    csa2.sparse_attn_decode(c, q.cuda(), q_pos, idx.cuda(), out2, lse2, ws, scale,
                            sink=sink.cuda() if sink is not None else None, err=err)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("swa_dtype", [csa2.SWA_BF16, csa2.SWA_MXFP8])
def test_sparse_attn_decode_large_window_values(orc, swa_dtype):
    """Latent rows scaled by 2^18 (the FP4 scales saturate, the window rows do not fit
    fp16) and the query by 2^-18: the window entries take a power-of-two scale 2^-sigma
    on the tensor-core path and the logits stay moderate."""
    B, T, H, k = 2, 400, 64, 256
    c, oc, _, err = build_r1(orc, B, T, swa_dtype, seed=71, kv_scale=2.0 ** 18)
    _, _, q = _decode_inputs(B, 4, H, seed=72)
    q = (q.float() * 2.0 ** -18).to(torch.bfloat16)
    g = torch.Generator().manual_seed(73)
    idx = torch.stack([torch.sort(torch.randperm(T - 1, generator=g)[:k]).values for _ in range(B)]).to(torch.int32)
    q_pos = torch.full((B,), T - 1, dtype=torch.int64, device="cuda")
    out = torch.empty((B, H, 512), device="cuda")
    lse = torch.empty((B, H), device="cuda")
    scale = 1 / math.sqrt(576)
    csa2.sparse_attn_decode(c, q.cuda(), q_pos, idx.cuda(), out, lse, csa2.attn_workspace(B, H, k), scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for b in range(B):
        ro, rl = orc.sparse_attn(oc[b], u16(q[b]), idx[b].numpy(), T - 1, scale)
        attn_close(out[b].cpu().numpy(), lse[b].cpu().numpy(), ro, rl)


def test_attn_index_error_is_reported(orc):
    c, oc, _, err = build_r1(orc, 1, 50, csa2.SWA_MXFP8, seed=51)
    _, _, q = _decode_inputs(1, 4, 16, seed=52)
    idx = torch.tensor([[3, 49, 60, -1]], dtype=torch.int32)  # 49 and 60 are not visible at q_pos 49
    q_pos = torch.tensor([49], dtype=torch.int64, device="cuda")
    out = torch.empty((1, 16, 512), device="cuda")
    lse = torch.empty((1, 16), device="cuda")
    ws = csa2.attn_workspace(1, 16, 4)
    csa2.sparse_attn_decode(c, q.cuda(), q_pos, idx.cuda(), out, lse, ws, 0.05, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & csa2.DEVERR_INDEX
    ro, rl = orc.sparse_attn(oc[0], u16(q[0]), np.array([3, -1, -1, -1], np.int32), 49, 0.05)
    attn_close(out[0].cpu().numpy(), lse[0].cpu().numpy(), ro, rl)


# ------------------------------------------------------------------ one decode step (tiny workload)
def test_tiny_decode_step_end_to_end(orc):
    """Batch 1, context 4,096, 16 heads, 4 indexer heads, top-64, bf16 window:
    append the step's token, Full-layer score, top-k + pool, attention."""
    W = wl.tiny_decode()
    B, ctx = W.batch, W.context
    c, oc, rope, err = build_r1(orc, B, ctx + 1, W.swa_dtype, seed=W.seed, chunks=[ctx, 1],
                                cap=ctx + 64)
    q_idx, w, q = W.q_idx(0, 0), W.w(0, 0), W.q(0, 0)
    q_pos = torch.full((B,), ctx, dtype=torch.int64, device="cuda")
    scores = torch.empty((B, c.capacity), device="cuda")
    csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores, err=err)
    idx = torch.empty((B, W.topk), dtype=torch.int32, device="cuda")
    pool = torch.empty((B, 2048), dtype=torch.int32, device="cuda")
    pcnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = csa2.topk_workspace(B, c.capacity, W.topk, 2048)
    csa2.topk(scores, 1, q_pos, W.topk, idx, ws, pool_out=pool, pool_count=pcnt, err=err)
    out = torch.empty((B, W.heads, 512), device="cuda")
    lse = torch.empty((B, W.heads), device="cuda")
    aws = csa2.attn_workspace(B, W.heads, W.topk)
    csa2.sparse_attn_decode(c, q.cuda(), q_pos, idx, out, lse, aws, W.sm_scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    r_idx, r_pool, r_cnt, r_out, r_lse, r_scores = orc.full_layer(
        oc[0], u16(q_idx[0]), w[0].numpy(), u16(q[0]), ctx, W.topk, W.sm_scale)
    assert np.array_equal(scores[0, :ctx].cpu().numpy().view(np.uint32), r_scores.view(np.uint32))
    assert idx[0].tolist() == r_idx.tolist()
    assert pcnt[0].item() == r_cnt == 512 and pool[0].tolist() == r_pool.tolist()
    attn_close(out[0].cpu().numpy(), lse[0].cpu().numpy(), r_out, r_lse)


def test_encoder_group_decode_steps(orc):
    """Encoder-style group at decode (ratio 2): every step appends one token per
    sequence through the compression buffer (an entry completes every second step,
    the prior length is odd so the first step completes one), then a Full layer over
    the visible entries (with the sideband, no pool) and two Reuse layers with their
    own queries.  Cache bytes and indices exact, attention within tolerance."""
    B, prior, steps, H_I, H, k, seed = 2, 601, 4, 4, 16, 32, 71
    c, oc, rope, err, (ba, bb), _, _ = build_r2(orc, B, prior, csa2.SWA_MXFP8, seed=seed,
                                               cap=(prior + steps) // 2 + 8)
    scale = 1 / math.sqrt(576)
    g = torch.Generator().manual_seed(72)
    scores = torch.empty((B, c.capacity), device="cuda")
    aux = csa2.score_aux(B, c.capacity)
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    out = torch.empty((B, H, 512), device="cuda")
    lse = torch.empty((B, H), device="cuda")
    ws_t = csa2.topk_workspace(B, c.capacity, k)
    ws_a = csa2.attn_workspace(B, H, k)
    for s in range(steps):
        t = prior + s
        rows = [torch.stack(x) for x in zip(*[cmp_rows(seed, b, t, 1) for b in range(B)])]
        csa2.kv_append(c, rope_cs=rope, cmp=[r.cuda() for r in rows] + [ba.cuda(), bb.cuda()], err=err)
        for b in range(B):
            orc.append_r2(oc[b], *[r[b].numpy() for r in rows], ba.numpy(), bb.numpy(), 1e4)
        q_pos = torch.full((B,), t, dtype=torch.int64, device="cuda")
        q_idx = torch.randn((B, H_I, 128), generator=g).to(torch.bfloat16)
        w = torch.rand((B, H_I), generator=g)
        qs = [torch.randn((B, H, 576), generator=g).to(torch.bfloat16) for _ in range(3)]
        csa2.index_score(c, q_idx.cuda(), w.cuda(), q_pos, scores, err=err, aux=aux)
        csa2.topk(scores, 2, q_pos, k, idx, ws_t, err=err, aux=aux)
        r_idx = []
        for layer in range(3):
            csa2.sparse_attn_decode(c, qs[layer].cuda(), q_pos, idx, out, lse, ws_a, scale, err=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            for b in range(B):
                if layer == 0:
                    ri, _, _, ro, rl, _ = orc.full_layer(oc[b], u16(q_idx[b]), w[b].numpy(), u16(qs[0][b]), t, k,
                                                         scale)
                    assert idx[b].tolist() == ri.tolist(), f"step {s} sequence {b}"
                    r_idx.append(ri)
                else:
                    ro, rl = orc.reuse_layer(oc[b], u16(qs[layer][b]), t, r_idx[b], scale)
                attn_close(out[b].cpu().numpy(), lse[b].cpu().numpy(), ro, rl)
    assert c.n_tokens.tolist() == [prior + steps] * B
    assert_cache_equal(c, oc, (prior + steps) // 2)


# ------------------------------------------------------------------ prefill (small)
@pytest.mark.parametrize("prior,Q,H_I,H,use_sink", [
    (300, 70, 4, 16, False),
    (300, 71, 64, 16, False),   # 64 indexer heads (the workloads' count), an odd chunk
    (301, 40, 64, 16, False),   # odd prior: a token waits in the compression buffer
    (301, 33, 16, 96, True),    # two head blocks of the attention (64 + 32 padded), with a sink
])
def test_prefill_chunk_small(orc, prior, Q, H_I, H, use_sink):
    k = 32
    c, oc, rope, err, (ba, bb), _, _ = build_r2(orc, 2, prior, csa2.SWA_MXFP8, seed=61,
                                               chunks=[prior], cap=(prior + Q) // 2 + 8)
    seq = 1
    rows = cmp_rows(61, seq, prior, Q)  # C^a, C^b, Z^a, Z^b rows [Q, 704] of the chunk
    g = torch.Generator().manual_seed(62)
    q_idx = torch.randn((Q, H_I, 128), generator=g).to(torch.bfloat16)
    w = torch.rand((Q, H_I), generator=g)
    q = torch.randn((Q, H, 576), generator=g).to(torch.bfloat16)
    sink = (torch.randn((H,), generator=g) * 2).float() if use_sink else None
    idx = torch.empty((Q, k), dtype=torch.int32, device="cuda")
    out = torch.empty((Q, H, 512), device="cuda")
    lse = torch.empty((Q, H), device="cuda")
    ws = csa2.prefill_workspace(Q, c.capacity, H_I, H, k)
    scale = 1 / math.sqrt(576)
    csa2.prefill_chunk(c, seq, [r.cuda() for r in rows] + [ba.cuda(), bb.cuda()], rope, q_idx.cuda(),
                       w.cuda(), q.cuda(), k, scale, idx, out, lse, ws,
                       sink=sink.cuda() if sink is not None else None, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o = oc[seq]
    # window rows of the prior tokens as they were before the chunk (the ring)
    prior_ring = {t: (o.swa_codes[t % 128].copy(), o.swa_scales[t % 128].copy())
                  for t in range(max(0, prior - 128), prior)}
    orc.append_r2(o, *[r.numpy() for r in rows], ba.numpy(), bb.numpy(), 1e4)
    # the appended chunk: cache bytes of this sequence match
    n_e = (prior + Q) // 2
    for name in ("lat_codes", "rope_codes"):
        assert np.array_equal(getattr(c, name)[seq, :n_e].cpu().numpy(), getattr(o, name)[:n_e])
    assert np.array_equal(c.idx_entries()[0][seq, :n_e].cpu().numpy(), o.idx_codes[:n_e])
    chunk_win = {}
    for i in range(Q):
        t = prior + i
        chunk_win[t] = orc.encode_swa(rows[0][i, :576].numpy(), orc.rope_cs(1e4, t), csa2.SWA_MXFP8)
    for i in range(Q):
        t = prior + i
        T = t // 2
        sc, flags = orc.index_scores(o, u16(q_idx[i]), w[i].numpy(), n_vis=T)
        assert flags == 0
        r_idx = orc.topk(sc, k)
        assert idx[i].tolist() == r_idx.tolist(), f"query {i}"
        toks = list(range(max(0, t - 127), t + 1))
        wc = np.array([(chunk_win[x] if x >= prior else prior_ring[x])[0] for x in toks])
        wsc = np.array([(chunk_win[x] if x >= prior else prior_ring[x])[1] for x in toks])
        ro, rl = orc.sparse_attn(o, u16(q[i]), r_idx, t, scale, sink=sink.numpy() if sink is not None else None,
                                 swa_codes=wc, swa_scales=wsc)
        attn_close(out[i].cpu().numpy(), lse[i].cpu().numpy(), ro, rl)
