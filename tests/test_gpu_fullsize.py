"""Parity at the workloads' full sizes, in the launch shapes bench.py times.

Every index score of the checked rows is compared with the oracle: the oracle
encodes the indexer key of every visible position from the same seeded rows
(the MXFP4 key records alone, which is all the score reads), scores the whole
row, and its own top-k and candidate pool are the references for the GPU's
selection.  The oracle never reads a GPU result.  Latent records are checked
at sampled positions and at every selected one, and attention outputs within
2e-3 normwise of the oracle's fp64 attention over the oracle-selected entries
and the window.
"""
import numpy as np
import pytest
import torch

from fp4_compressed_sparse_gb300 import csa2
from fp4_compressed_sparse_gb300 import workloads as wl
from gpu_util import attn_close, u16
from fullsize_util import (CHUNK, Compact, assert_entries_equal, build_gpu_r1, oracle_keys,
                           window_records)

pytestmark = pytest.mark.gpu
SAMPLE = 4096


def _sample(rng, T, extra):
    s = rng.choice(T, size=min(SAMPLE, T), replace=False)
    return np.unique(np.concatenate([s, np.asarray(extra, np.int64)[np.asarray(extra) >= 0],
                                     np.arange(max(0, T - 8), T)]))


def _check_full_layer(orc, W, c, seq, q_pos, q_idx, w, q, scores, idx, pool, pool_cnt, out, lse, rng):
    """Whole-row check of one Full layer of sequence `seq`: key records and scores
    of every visible position bit-exact, top-k and pool equal to the oracle's
    selection over its own scores, attention within 2e-3."""
    T = q_pos  # ratio 1: entries 0 .. q_pos-1 are visible
    kc = oracle_keys(orc, W, seq, T)
    ic, isc = c.idx_entries()
    assert np.array_equal(ic[seq, :T].cpu().numpy(), kc.idx_codes), f"seq {seq}: key codes"
    assert np.array_equal(isc[seq, :T].cpu().numpy(), kc.idx_scales), f"seq {seq}: key scales"
    ref, flags = orc.index_scores(kc, u16(q_idx[seq]), w[seq].cpu().numpy(), n_vis=T)
    assert flags == 0
    got = scores[seq, :T].cpu().numpy()
    bad = np.nonzero(got.view(np.uint32) != ref.view(np.uint32))[0]
    assert bad.size == 0, f"seq {seq}: {bad.size} of {T} scores differ, first at {bad[:4].tolist()}"
    k = idx.shape[1]
    r_idx = orc.topk(ref, k)
    g_idx = idx[seq].cpu().numpy()
    assert g_idx.tolist() == r_idx.tolist(), f"seq {seq}: top-k"
    if pool is not None:
        pids, cnt = orc.pool(ref, T, 8, pool.shape[1])
        assert int(pool_cnt[seq].item()) == cnt, f"seq {seq}: pool count"
        assert pool[seq].cpu().numpy().tolist() == pids.tolist(), f"seq {seq}: pool"
    comp = Compact(orc, W, seq, _sample(rng, T, r_idx))
    assert_entries_equal(c, seq, comp)
    wc, wsc = window_records(orc, W, seq, q_pos, q_pos + 1)
    ro, rl = orc.sparse_attn(comp.cache, u16(q[seq]), comp.remap(r_idx), q_pos, W.sm_scale,
                             swa_codes=wc, swa_scales=wsc)
    attn_close(out[seq].cpu().numpy(), lse[seq].cpu().numpy(), ro, rl)


def test_full_decode_b32_t65536(orc):
    """Full-layer decode, batch 32, context 65,536, 64 heads, 64 indexer heads,
    top-512 + 2,048-block pool, MXFP8 window: one bench step."""
    import bench
    W = wl.full_decode(device="cuda")
    fd = bench.FullDecode(W, 1, torch.device("cuda"))
    fd.step(0)
    torch.cuda.synchronize()
    assert int(fd.err.item()) == 0
    rng = np.random.default_rng(11)
    for seq in (0, 17):
        _check_full_layer(orc, W, fd.cache, seq, W.context, fd.q_idx[0], fd.w[0], fd.q[0], fd.scores,
                          fd.idx, fd.pool, fd.pool_cnt, fd.out, fd.lse, rng)


def _append_step_token(W, c, rope, err, step):
    t = W.context + step
    kv = torch.stack([W.kv(b, t, 1, device="cuda") for b in range(W.batch)])
    ik = torch.stack([W.ik(b, t, 1, device="cuda") for b in range(W.batch)])
    csa2.kv_append(c, kv, ik, rope, err=err)
    return torch.full((W.batch,), t, dtype=torch.int64, device="cuda")


def _reindex_and_reuse(orc, W, c, q_pos, pool_dev, layers, seqs, leader_layer, err, rng):
    """Run `layers` (Reindex / Reuse) on the GPU from a pool, check seqs."""
    B, k = W.batch, W.topk
    stride = pool_dev.shape[1] * W.pool_block_size
    scores = torch.empty((B, stride), device="cuda")
    aux = csa2.score_aux(B, stride)
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    out = torch.empty((B, W.heads, 512), device="cuda")
    lse = torch.empty((B, W.heads), device="cuda")
    ws_t = csa2.topk_workspace(B, stride, k)
    ws_a = csa2.attn_workspace(B, W.heads, k)
    results = []
    for li, role in enumerate(layers):
        layer = leader_layer + li
        if role == "reindex":
            q_idx, w = W.q_idx(0, layer), W.w(0, layer)
            csa2.index_score(c, q_idx, w, q_pos, scores, pool=pool_dev, err=err, aux=aux)
            csa2.topk(scores, 1, q_pos, k, idx, ws_t, pool=pool_dev, err=err, aux=aux)
            last = (q_idx, w, scores.clone(), idx.clone())
        q = W.q(0, layer)
        csa2.sparse_attn_decode(c, q, q_pos, idx, out, lse, ws_a, W.sm_scale, err=err)
        results.append((role, last, q, out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for seq in seqs:
        qp = int(q_pos[seq].item())
        pids = pool_dev[seq].cpu().numpy()
        cnt = int((pids >= 0).sum())
        pos = orc.pool_positions(pids, cnt, qp, W.pool_block_size)
        comp = Compact(orc, W, seq, pos)
        assert_entries_equal(c, seq, comp)
        wc, wsc = window_records(orc, W, seq, qp, qp + 1)
        for role, (q_idx, w, sc, ix), q, o, l in results:
            g_idx = ix[seq].cpu().numpy()
            if role == "reindex":
                ref, flags = orc.index_scores(comp.cache, u16(q_idx[seq]), w[seq].cpu().numpy(),
                                              n_vis=comp.positions.shape[0])
                assert flags == 0
                # slot j of the score row is position pool[j // 8] * 8 + j % 8
                slots = np.array([list(pids[:cnt]).index(p // 8) * 8 + p % 8 for p in pos])
                got = sc[seq].cpu().numpy()[slots]
                assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"seq {seq} reindex scores"
                assert g_idx.tolist() == orc.topk(ref, W.topk, positions=pos).tolist(), f"seq {seq} reindex top-k"
            ro, rl = orc.sparse_attn(comp.cache, u16(q[seq]), comp.remap(g_idx), qp, W.sm_scale,
                                     swa_codes=wc, swa_scales=wsc)
            attn_close(o[seq].cpu().numpy(), l[seq].cpu().numpy(), ro, rl)


def test_reindex_reuse3_b64_t262144(orc):
    """Reindex-layer decode, batch 64, context 262,144: scoring inside a prior pool of
    2,048 uniformly drawn blocks x 8, top-512, then 3 Reuse layers."""
    W = wl.reindex_decode(device="cuda")
    c, rope, err = build_gpu_r1(W)
    q_pos = _append_step_token(W, c, rope, err, 0)
    pool_dev = W.pool(device="cuda")
    _reindex_and_reuse(orc, W, c, q_pos, pool_dev, W.layers, (0, 41), 0, err,
                       np.random.default_rng(12))


def test_stack_b8_t1048576_one_step(orc):
    """Long-context decoder group at batch 8, context 1,048,576: one step of append,
    Full (scan + pool), 4 Reindex, 3 Reuse."""
    W = wl.stack_1m(device="cuda")
    c, rope, err = build_gpu_r1(W)
    q_pos = _append_step_token(W, c, rope, err, 0)
    B, k = W.batch, W.topk
    stride = c.capacity
    scores = torch.empty((B, stride), device="cuda")
    aux = csa2.score_aux(B, stride)
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    pool = torch.empty((B, W.pool_blocks), dtype=torch.int32, device="cuda")
    pcnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    out = torch.empty((B, W.heads, 512), device="cuda")
    lse = torch.empty((B, W.heads), device="cuda")
    q_idx, w, q = W.q_idx(0, 0), W.w(0, 0), W.q(0, 0)
    csa2.index_score(c, q_idx, w, q_pos, scores, err=err, aux=aux)
    csa2.topk(scores, 1, q_pos, k, idx, csa2.topk_workspace(B, stride, k, W.pool_blocks), pool_out=pool,
              pool_count=pcnt, err=err, aux=aux)
    csa2.sparse_attn_decode(c, q, q_pos, idx, out, lse, csa2.attn_workspace(B, W.heads, k), W.sm_scale,
                            err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rng = np.random.default_rng(13)
    _check_full_layer(orc, W, c, 0, W.context, q_idx, w, q, scores, idx, pool, pcnt, out, lse, rng)
    _reindex_and_reuse(orc, W, c, q_pos, pool, W.layers[1:], (0,), 1, err, rng)


def test_prefill_q8192_prior131072(orc):
    """Encoder-style chunked prefill: 8,192 query tokens against 131,072 prior tokens
    packed 2 per entry (65,536 entries), 64 indexer heads, top-512, 64 heads, MXFP8
    window.  The cache is compared whole; the first and last query of every score
    block and of every 512-query span (49 queries) are checked against full
    oracle scans."""
    W = wl.prefill_chunk(device="cuda")
    cap = (W.prior + W.chunk) // 2 + 8
    c = csa2.Cache(1, cap, ratio=2, swa_dtype=W.swa_dtype)
    rope = csa2.rope_table(W.theta, 2 * cap + 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ba, bb = W.bias(device="cuda")
    for t0 in range(0, W.prior, wl.CHUNK):
        rows = W.cmp_rows(t0, wl.CHUNK, device="cuda")
        csa2.kv_append(c, rope_cs=rope, cmp=[r[None] for r in rows] + [ba, bb], err=err)
    rows = W.cmp_rows(W.prior, W.chunk, device="cuda")
    q_idx, w, q = W.q_idx(device="cuda"), W.w(device="cuda"), W.q(device="cuda")
    Q, k = W.chunk, W.topk
    idx = torch.empty((Q, k), dtype=torch.int32, device="cuda")
    out = torch.empty((Q, W.heads, 512), device="cuda")
    lse = torch.empty((Q, W.heads), device="cuda")
    ws = csa2.prefill_workspace(Q, cap, W.index_heads, W.heads, k)
    csa2.prefill_chunk(c, 0, list(rows) + [ba, bb], rope, q_idx, w, q, k, W.sm_scale, idx, out, lse, ws,
                       err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    # the oracle's cache of the whole sequence, entry by entry from the same rows
    n_entries = (W.prior + W.chunk) // 2
    o = orc.Cache(n_entries, swa_dtype=W.swa_dtype, ratio=2)
    zb = np.zeros((2, 704), np.float32)
    prev = None  # the last two tokens' rows of the previous chunk
    for t0 in range(0, W.prior + W.chunk, wl.CHUNK):
        ca, cb, za, zbr = (r.cpu().numpy() for r in W.cmp_rows(t0, wl.CHUNK, device="cuda"))
        for j in range(0, wl.CHUNK, 2):
            i = (t0 + j) // 2
            if j >= 2:
                b_rows = (cb[j - 2:j], zbr[j - 2:j])
            elif prev is not None:
                b_rows = prev
            else:
                b_rows = None
            v = orc.compress_entry(2, [ca[j], ca[j + 1]], [za[j], za[j + 1]],
                                   list(b_rows[0]) if b_rows else None, list(b_rows[1]) if b_rows else None,
                                   zb, zb)
            rec = orc.encode_entry(v[:576], v[576:], orc.rope_cs(W.theta, 2 * i))
            for arr, val in zip((o.lat_codes, o.lat_scales, o.rope_codes, o.rope_scales, o.idx_codes,
                                 o.idx_scales), rec):
                arr[i] = val
        prev = (cb[-2:], zbr[-2:])
    o.n_tokens = W.prior + W.chunk
    o.n_entries = n_entries
    ic, isc = c.idx_entries()
    for name, g in (("lat_codes", c.lat_codes), ("lat_scales", c.lat_scales), ("rope_codes", c.rope_codes),
                    ("rope_scales", c.rope_scales), ("idx_codes", ic), ("idx_scales", isc)):
        assert np.array_equal(g[0, :n_entries].cpu().numpy(), getattr(o, name)), f"prefill cache {name}"
    # the chunk is scored in blocks of queries whose fp32 score rows fill 256 MB,
    # rounded down to a multiple of twice the SM count: the first and last query
    # of every such block, of every 512-query span, and the middle of the chunk
    qb = (256 << 20) // (cap * 4)
    wave = 2 * torch.cuda.get_device_properties(0).multi_processor_count
    if qb > wave:
        qb = qb // wave * wave
    qb = max(1, min(Q, 4096, qb))
    qs = {1, Q // 2 - 1, Q // 2}
    for span in (qb, 512):
        for q0 in range(0, Q, span):
            qs.update((q0, min(Q, q0 + span) - 1))
    qs = sorted(qs)
    assert len(qs) >= 16
    for i in qs:
        t = W.prior + i
        sc, flags = orc.index_scores(o, u16(q_idx[i]), w[i].cpu().numpy(), n_vis=t // 2)
        assert flags == 0
        r_idx = orc.topk(sc, k)
        assert idx[i].cpu().numpy().tolist() == r_idx.tolist(), f"query {i} top-k"
        toks = list(range(max(0, t - 127), t + 1))
        ca_w = np.zeros((len(toks), 576), np.float32)
        blks = {}
        for j, tok in enumerate(toks):
            ch = tok // wl.CHUNK
            if ch not in blks:
                blks[ch] = W.cmp_rows(ch * wl.CHUNK, wl.CHUNK, device="cuda")[0].cpu().numpy()
            ca_w[j] = blks[ch][tok - ch * wl.CHUNK, :576]
        recs = [orc.encode_swa(ca_w[j], orc.rope_cs(W.theta, tok), W.swa_dtype) for j, tok in enumerate(toks)]
        ro, rl = orc.sparse_attn(o, u16(q[i]), r_idx, t, W.sm_scale, swa_codes=np.array([r[0] for r in recs]),
                                 swa_scales=np.array([r[1] for r in recs]))
        attn_close(out[i].cpu().numpy(), lse[i].cpu().numpy(), ro, rl)
