"""Pins of the oracle's method steps (C4 score, C6 top-k, C7 pool, C8 attention,
C9 RoPE, C10 compression, visibility and the pages' byte accounting).

Brute force here is an independent route: exact rational arithmetic
(fractions.Fraction) with an explicit round-to-nearest-even to fp32, numpy's
float64 softmax, Python's sorted(), and the numbers printed on the pages.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

GOLD = os.path.join(os.path.dirname(__file__), "golden")
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ------------------------------------------------------------ helpers (independent)
def dec_e2m1(c):
    v = E2M1[c & 7]
    return -v if c & 8 else v


def dec_e4m3(c):
    s, e, m = c >> 7, (c >> 3) & 15, c & 7
    v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if s else v


def unpack(codes):
    out = []
    for b in codes:
        out += [int(b) & 15, int(b) >> 4]
    return out


def mx4_values(codes, scales):
    c = unpack(codes)
    return [Fraction(dec_e2m1(c[i])) * Fraction(2) ** (int(scales[i // 32]) - 127)
            for i in range(len(c))]


def nv4_values(codes, scales):
    c = unpack(codes)
    return [dec_e2m1(c[i]) * dec_e4m3(int(scales[i // 16])) for i in range(len(c))]


def bits32(f):
    return int(np.array([f], np.float32).view(np.uint32)[0])


def round_f32(x: Fraction) -> np.float32:
    f = np.float32(float(x))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda c: (abs(Fraction(float(c)) - x), bits32(c) & 1))


def fmaf(a, b, c):
    return round_f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def bf16(x):
    import torch
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def make_cache(orc, T, rng, swa_dtype=1, theta=10000.0):
    c = orc.Cache(T + 8, swa_dtype=swa_dtype)
    kv = rng.standard_normal((T, 576)).astype(np.float32)
    ik = rng.standard_normal((T, 128)).astype(np.float32)
    orc.append_r1(c, kv, ik, theta)
    return c, kv, ik


# ------------------------------------------------------------ accounting (pages)
def _gold(name):
    rows = {}
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                parts = line.split()
                rows.setdefault(parts[0], []).append(parts[1:])
    return rows


def test_accounting_matches_pages(orc):
    g = {k: float(v[0][0]) for k, v in _gold("accounting.txt").items()}
    c = orc.Cache(4)
    main = c.lat_codes.shape[1] + c.lat_scales.shape[1]
    idx = c.idx_codes.shape[1] + c.idx_scales.shape[1]
    assert main == g["main_entry_bytes"] == orc.lib().orc_main_entry_bytes(512, 16)
    assert idx == g["indexer_entry_bytes"] == orc.lib().orc_mx_entry_bytes(128, 32)
    assert main + idx == g["entry_total_bytes"]
    assert (main + idx) / 2 == g["encoder_bytes_per_token"]
    per_tok = 3 * (main + idx) / 2 + (main + idx)
    assert per_tok == g["global_bytes_per_token"]
    all_full = 18 * (main + idx) / 2 + 20 * (main + idx)
    assert all_full == g["all_full_bytes_per_token"]
    assert round(all_full / per_tok, 1) == g["all_full_ratio"]
    # the pages print these rounded to the digits shown (111.25 -> "about 111.3")
    assert abs(per_tok * 131072 / 2 ** 20 - g["mib_at_131072_tokens"]) <= 0.05
    assert abs(per_tok * 2 ** 20 / 2 ** 30 - g["gib_at_1048576_tokens"]) <= 0.0005
    assert abs(per_tok * 32 * 2 ** 20 / 2 ** 30 - g["gib_at_32x1048576"]) <= 0.05
    assert 448 * 6 == g["fp4_max_with_scale"]
    assert g["pool_blocks"] * g["pool_block_size"] == g["pool_positions"]


def test_layer_roles_reproduce_890(orc):
    """Role masks over the layer table: a layer with compression ratio 0 keeps
    only its window; among the others the KV-source ids hold a global cache
    (Full), the further index-source ids only re-score (Reindex) and the rest
    reuse.  The global bytes per token sum the Full layers' records divided by
    their ratios."""
    g = _gold("layer_roles.txt")
    n_layers = int(g["num_hidden_layers"][0][0])
    ratios = np.concatenate([np.full(int(n), int(v)) for v, n in
                             (run.split("x") for run in g["compress_ratios_runs"][0])])
    ids = np.arange(n_layers)
    compressed = ratios[:n_layers] > 0
    full = compressed & np.isin(ids, [int(x) for x in g["kv_source_layer_ids"][0]])
    reindex = compressed & ~full & np.isin(ids, [int(x) for x in g["index_source_layer_ids"][0]])
    reuse = compressed & ~full & ~reindex
    c = orc.Cache(4)
    record = sum(a.shape[1] for a in (c.lat_codes, c.lat_scales, c.idx_codes, c.idx_scales))
    per_token = float(np.sum(record / ratios[:n_layers][full]))
    want = {e[0]: e[1] for e in g["expect"]}
    counts = {"swa-only": int(np.sum(~compressed)), "full": int(full.sum()), "reindex": int(reindex.sum()),
              "reuse": int(reuse.sum())}
    assert counts == {k: int(want[k]) for k in counts}
    assert ratios.shape[0] == int(want["compress_ratios_entries"])
    assert per_token == float(want["global_bytes_per_token"])


def test_encode_keys_equals_entry_records(orc):
    """The key-only encoder gives the indexer planes of the full entry encoder."""
    rng = np.random.default_rng(41)
    n = 300
    kv = rng.standard_normal((n, 576)).astype(np.float32)
    ik = (rng.standard_normal((n, 128)) * 2.0 ** rng.integers(-20, 20, (n, 1))).astype(np.float32)
    ik[5] = 0.0
    full = orc.Cache(n)
    orc.append_r1(full, kv, ik, 1e4)
    keys = orc.KeyCache(n + 7)
    orc.encode_keys(keys, 7, ik)
    assert np.array_equal(keys.idx_codes[7:], full.idx_codes[:n])
    assert np.array_equal(keys.idx_scales[7:], full.idx_scales[:n])
    assert not keys.idx_codes[:7].any()


# ------------------------------------------------------------ RoPE (C9)
def test_rope_pos0_identity_and_norm(orc):
    rng = np.random.default_rng(1)
    x = rng.standard_normal(64).astype(np.float32)
    assert np.array_equal(orc.rope_apply(x, orc.rope_cs(10000.0, 0)), x)
    for pos in (1, 17, 4096, 65535, 1048575):
        y = orc.rope_apply(x, orc.rope_cs(10000.0, pos))
        n0 = np.hypot(x[0::2].astype(np.float64), x[1::2])
        n1 = np.hypot(y[0::2].astype(np.float64), y[1::2])
        assert np.allclose(n0, n1, rtol=4e-7, atol=1e-7)


def test_rope_relative_phase(orc):
    # [P2] §3: the rotated q.k depends on the distance t - s only
    rng = np.random.default_rng(2)
    q = rng.standard_normal(64).astype(np.float32)
    k = rng.standard_normal(64).astype(np.float32)

    def dot(t, s):
        return float(np.dot(orc.rope_apply(q, orc.rope_cs(1e4, t)).astype(np.float64),
                            orc.rope_apply(k, orc.rope_cs(1e4, s))))

    assert dot(100, 40) == pytest.approx(dot(1060, 1000), rel=1e-4, abs=1e-4)
    assert dot(7, 7) == pytest.approx(float(np.dot(q.astype(np.float64), k)), rel=1e-4, abs=1e-4)


def test_rope_pairs_interleaved(orc):
    # a vector that is nonzero only in pair 0 stays inside pair 0 and turns by pos * theta^0
    x = np.zeros(64, np.float32)
    x[0] = 1.0
    y = orc.rope_apply(x, orc.rope_cs(1e4, 3))
    assert np.all(y[2:] == 0)
    assert y[0] == np.float32(math.cos(3.0)) and y[1] == np.float32(math.sin(3.0))
    # pair i uses theta^(-2i/64)
    x = np.zeros(64, np.float32)
    x[2 * 5] = 1.0
    y = orc.rope_apply(x, orc.rope_cs(1e4, 9))
    assert y[10] == np.float32(math.cos(9 * 1e4 ** (-10 / 64)))


# ------------------------------------------------------------ entry encode
def test_entry_encode_roundtrip(orc):
    rng = np.random.default_rng(4)
    v = rng.standard_normal(576).astype(np.float32)
    ik = rng.standard_normal(128).astype(np.float32)
    cs = orc.rope_cs(1e4, 123)
    lc, ls, rc, rs, ic, isc = orc.encode_entry(v, ik, cs)
    lat = np.array(nv4_values(lc, ls))
    assert np.max(np.abs(lat - v[:512])) < 0.6  # one half-step of a scale <= 3.75/6*... bound
    r = orc.rope_apply(v[512:], cs)
    rope = np.array(nv4_values(rc, rs))
    assert np.max(np.abs(rope - r)) < 0.6
    idx = np.array([float(x) for x in mx4_values(ic, isc)])
    assert np.max(np.abs(idx - ik)) < 0.6
    # the unrotated rope dims must NOT match as well as the rotated ones (quantise after RoPE)
    assert np.max(np.abs(rope - v[512:])) > 0.6


# ------------------------------------------------------------ index score (C4)
def test_index_score_bruteforce_exact(orc):
    rng = np.random.default_rng(5)
    T, H = 40, 3
    cache, _, _ = make_cache(orc, T, rng)
    q = bf16(rng.standard_normal((H, 128)))
    w = rng.uniform(-1, 1, H).astype(np.float32)
    got, flags = orc.index_scores(cache, q, w, n_vis=T)
    assert flags == 0
    qc = np.zeros((H, 64), np.uint8)
    qs = np.zeros((H, 4), np.uint8)
    orc.lib().orc_quant_q_index(H, orc._p(np.ascontiguousarray(q)), orc._p(qc), orc._p(qs))
    qv = [mx4_values(qc[h], qs[h]) for h in range(H)]
    for s in range(T):
        kv = mx4_values(cache.idx_codes[s], cache.idx_scales[s])
        acc = np.float32(0.0)
        for h in range(H):
            d = round_f32(sum(a * b for a, b in zip(qv[h], kv)))
            r = d if d > 0 else np.float32(0.0)
            acc = fmaf(w[h], r, acc)
        assert bits32(got[s]) == bits32(acc), (s, got[s], acc)


def test_index_query_quantised_like_keys(orc):
    # the indexer query is quantised to MXFP4 with the same rule as the keys ([P5] §2.3.4)
    rng = np.random.default_rng(6)
    x = rng.standard_normal(128).astype(np.float32)
    xb = bf16(x)
    import torch
    xf = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).float().numpy()
    qc = np.zeros(64, np.uint8)
    qs = np.zeros(4, np.uint8)
    orc.lib().orc_quant_q_index(1, orc._p(np.ascontiguousarray(xb)), orc._p(qc), orc._p(qs))
    for b in range(4):
        c, s = orc.mxfp4_quant32(xf[32 * b:32 * b + 32])
        assert list(c) == list(qc[16 * b:16 * b + 16]) and s == qs[b]


def test_index_score_single_head_unit_weight_is_relu_dot(orc):
    rng = np.random.default_rng(8)
    T = 64
    cache, _, _ = make_cache(orc, T, rng)
    q = bf16(rng.standard_normal((1, 128)))
    got, _ = orc.index_scores(cache, q, np.ones(1, np.float32), n_vis=T)
    qc = np.zeros((1, 64), np.uint8)
    qs = np.zeros((1, 4), np.uint8)
    orc.lib().orc_quant_q_index(1, orc._p(np.ascontiguousarray(q)), orc._p(qc), orc._p(qs))
    qv = np.array([float(v) for v in mx4_values(qc[0], qs[0])])
    K = np.array([[float(v) for v in mx4_values(cache.idx_codes[s], cache.idx_scales[s])]
                  for s in range(T)])
    ref = np.maximum(K @ qv, 0.0).astype(np.float32)
    assert np.array_equal(got, ref)


def test_index_score_zero_weight_gives_lowest_positions(orc):
    rng = np.random.default_rng(9)
    T = 100
    cache, _, _ = make_cache(orc, T, rng)
    q = bf16(rng.standard_normal((4, 128)))
    got, _ = orc.index_scores(cache, q, np.zeros(4, np.float32), n_vis=T)
    assert not got.any()
    assert list(orc.topk(got, 10)) == list(range(10))


# ------------------------------------------------------------ top-k (C6)
@pytest.mark.parametrize("T,k", [(1, 4), (5, 5), (64, 8), (1000, 64), (4096, 512)])
def test_topk_bruteforce_with_ties(orc, T, k):
    rng = np.random.default_rng(T + k)
    s = rng.integers(0, 7, T).astype(np.float32) * np.float32(0.5)  # many ties
    s[rng.integers(0, T, max(1, T // 10))] = -0.0
    got = orc.topk(s, k)
    ref = sorted(range(T), key=lambda i: (-float(s[i]), i))[:k]
    want = sorted(ref) + [-1] * (k - min(k, T))
    assert list(got) == want


def test_topk_and_pool_with_infinities(orc):
    """-inf is an ordinary lowest score and +inf an ordinary highest one: rows with
    fewer finite scores than k, with more +inf scores than k, and mixed, against
    Python's sort on (score desc, position asc) and the block maxima it implies."""
    rng = np.random.default_rng(21)
    T, k, nb_keep = 600, 64, 16
    rows = []
    a = rng.standard_normal(T).astype(np.float32)
    a[30:] = -np.inf
    rows.append(a)
    b = rng.standard_normal(T).astype(np.float32)
    b[rng.choice(T, 100, replace=False)] = np.inf
    rows.append(b)
    c = rng.standard_normal(T).astype(np.float32)
    c[rng.choice(T, 7, replace=False)] = np.inf
    c[rng.choice(T, 200, replace=False)] = -np.inf
    rows.append(c)
    rows.append(np.full(T, -np.inf, np.float32))
    for s in rows:
        ref = sorted(sorted(range(T), key=lambda i: (-float(s[i]), i))[:k])
        assert list(orc.topk(s, k)) == ref
        nb = (T + 7) // 8
        bm = [max(float(x) for x in s[j * 8:min(T, j * 8 + 8)]) for j in range(nb)]
        ids, cnt = orc.pool(s, T, 8, nb_keep)
        assert cnt == nb_keep and list(ids) == sorted(sorted(range(nb), key=lambda j: (-bm[j], j))[:nb_keep])


def test_topk_positions_and_nan(orc):
    s = np.array([1.0, 3.0, 3.0, 2.0], np.float32)
    pos = np.array([40, 7, 9, 100])
    assert list(orc.topk(s, 2, positions=pos)) == [7, 9]
    with pytest.raises(ValueError):
        orc.topk(np.array([1.0, np.nan], np.float32), 1)


# ------------------------------------------------------------ pool (C7)
def test_pool_bruteforce(orc):
    rng = np.random.default_rng(12)
    T = 1000
    s = rng.integers(0, 50, T).astype(np.float32)
    ids, cnt = orc.pool(s, T, 8, 20)
    nb = (T + 7) // 8
    bm = [max(s[b * 8:min(T, b * 8 + 8)]) for b in range(nb)]
    ref = sorted(sorted(range(nb), key=lambda b: (-bm[b], b))[:20])
    assert cnt == 20 and list(ids) == ref


def test_pool_covers_everything_when_small(orc):
    T = 16384 - 5
    s = np.random.default_rng(0).standard_normal(T).astype(np.float32)
    ids, cnt = orc.pool(s, T)
    assert cnt == math.ceil(T / 8) and list(ids[:cnt]) == list(range(cnt))
    assert np.all(ids[cnt:] == -1)


def test_full_topk_inside_pool_and_reindex_equals_full(orc):
    rng = np.random.default_rng(13)
    T, H = 6000, 4
    cache, _, _ = make_cache(orc, T, rng)
    q_idx = bf16(rng.standard_normal((H, 128)))
    w = rng.uniform(0, 1, H).astype(np.float32)
    scores, _ = orc.index_scores(cache, q_idx, w, n_vis=T)
    k, nblk = 64, 100
    idx = orc.topk(scores, k)
    ids, cnt = orc.pool(scores, T, 8, nblk)
    pos = orc.pool_positions(ids, cnt, T)
    assert set(idx.tolist()) <= set(pos.tolist())
    s2, _ = orc.index_scores(cache, q_idx, w, rows=pos)
    assert list(orc.topk(s2, k, positions=pos)) == list(idx)


# ------------------------------------------------------------ attention (C8)
def _entries(cache, n):
    return np.array([nv4_values(cache.lat_codes[s], cache.lat_scales[s])
                     + nv4_values(cache.rope_codes[s], cache.rope_scales[s]) for s in range(n)])


def test_attention_dense_special_case(orc):
    rng = np.random.default_rng(14)
    T, H = 30, 5
    cache, _, _ = make_cache(orc, T, rng)
    q = bf16(rng.standard_normal((H, 576)))
    idx = np.arange(T, dtype=np.int32)
    scale = 1 / math.sqrt(576)
    out, lse = orc.sparse_attn(cache, q, idx, T - 1, scale, swa_codes=np.zeros((0, 576), np.uint8),
                               swa_scales=np.zeros((0, 18), np.uint8))
    import torch
    qf = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).double().numpy()
    E = _entries(cache, T)
    z = scale * (qf @ E.T)
    p = np.exp(z - z.max(1, keepdims=True))
    ref = (p @ E[:, :512]) / p.sum(1, keepdims=True)
    ref_lse = z.max(1) + np.log(p.sum(1))
    assert np.allclose(out, ref, rtol=1e-6, atol=1e-6)
    assert np.allclose(lse, ref_lse, rtol=1e-6, atol=1e-6)


def test_attention_single_entry_and_sink(orc):
    rng = np.random.default_rng(15)
    cache, _, _ = make_cache(orc, 10, rng)
    q = bf16(rng.standard_normal((2, 576)))
    none = dict(swa_codes=np.zeros((0, 576), np.uint8), swa_scales=np.zeros((0, 18), np.uint8))
    idx = np.array([4, -1, -1], np.int32)
    out, lse = orc.sparse_attn(cache, q, idx, 9, 0.05, **none)
    E = _entries(cache, 10)
    assert np.allclose(out, np.tile(E[4, :512], (2, 1)), rtol=1e-6, atol=1e-7)
    sink = np.array([0.3, -2.0], np.float32)
    out2, lse2 = orc.sparse_attn(cache, q, idx, 9, 0.05, sink=sink, **none)
    import torch
    qf = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).double().numpy()
    z = 0.05 * (qf @ E[4])
    frac = np.exp(z) / (np.exp(z) + np.exp(sink.astype(np.float64)))
    assert np.allclose(out2, frac[:, None] * E[4, :512][None], rtol=1e-6, atol=1e-7)
    assert np.allclose(lse2, np.log(np.exp(z) + np.exp(sink.astype(np.float64))), rtol=1e-6)
    assert np.all(frac < 1)


def test_attention_window_slots_and_reuse_identity(orc):
    rng = np.random.default_rng(16)
    T, H = 300, 4
    for swa_dtype in (0, 1):
        cache, kv, _ = make_cache(orc, T, rng, swa_dtype=swa_dtype)
        q = bf16(rng.standard_normal((H, 576)))
        idx = np.array([3, 77, 150, -1], np.int32)
        a = orc.sparse_attn(cache, q, idx, T - 1, 0.04)
        b = orc.sparse_attn(cache, q, idx, T - 1, 0.04)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        # the window holds tokens T-128..T-1 at slot t % 128; an MXFP8/bf16 copy of each
        toks = orc.swa_tokens(T - 1, T)
        assert toks == list(range(T - 128, T))
        for t in (T - 128, T - 1):
            cs = orc.rope_cs(1e4, t)
            c, s = orc.encode_swa(kv[t], cs, swa_dtype)
            assert np.array_equal(cache.swa_codes[t % 128], c)
            if swa_dtype == 1:
                assert np.array_equal(cache.swa_scales[t % 128], s)


# ------------------------------------------------------------ compression (C10)
def test_compress_uniform_gate_is_mean():
    from oracle import oracle as orc
    rng = np.random.default_rng(17)
    dim = 8
    rows = [rng.standard_normal(dim).astype(np.float32) for _ in range(4)]
    z = [np.full(dim, 0.7, np.float32)] * 4
    zero = np.zeros((2, dim), np.float32)
    v = orc.compress_entry(2, rows[2:], z[2:], rows[:2], z[:2], zero, zero)
    ref = np.mean(np.array(rows, np.float64), 0)
    assert np.allclose(v, ref, rtol=1e-6, atol=1e-7)
    v0 = orc.compress_entry(2, rows[2:], z[2:], None, None, zero, zero)  # entry 0: only a rows
    assert np.allclose(v0, np.mean(np.array(rows[2:], np.float64), 0), rtol=1e-6, atol=1e-7)


def test_compress_dominant_row_and_bias():
    from oracle import oracle as orc
    rng = np.random.default_rng(18)
    dim = 6
    rows = [rng.standard_normal(dim).astype(np.float32) for _ in range(4)]
    z = [np.zeros(dim, np.float32) for _ in range(4)]
    z[1] = np.full(dim, 200.0, np.float32)  # row b1 (token 2i-1) dominates
    zero = np.zeros((2, dim), np.float32)
    v = orc.compress_entry(2, rows[2:], z[2:], rows[:2], z[:2], zero, zero)
    assert np.allclose(v, rows[1], rtol=1e-6)
    ba = np.zeros((2, dim), np.float32)
    ba[0] = 300.0  # the positional bias of a-row 0 dominates
    v = orc.compress_entry(2, rows[2:], z[2:], rows[:2], z[:2], ba, zero)
    assert np.allclose(v, rows[2], rtol=1e-6)


def test_ratio2_entry_count_and_visibility(orc):
    rng = np.random.default_rng(19)
    c = orc.Cache(64, ratio=2)
    n = 21
    mk = lambda: rng.standard_normal((n, 704)).astype(np.float32)
    ba = rng.standard_normal((2, 704)).astype(np.float32)
    bb = rng.standard_normal((2, 704)).astype(np.float32)
    ca, cb, za, zb = mk(), mk(), mk(), mk()
    orc.append_r2(c, ca[:7], cb[:7], za[:7], zb[:7], ba, bb, 1e4)
    orc.append_r2(c, ca[7:], cb[7:], za[7:], zb[7:], ba, bb, 1e4)
    assert c.n_tokens == 21 and c.n_entries == 10  # 2 tokens per entry; token 20 pending
    c2 = orc.Cache(64, ratio=2)
    orc.append_r2(c2, ca, cb, za, zb, ba, bb, 1e4)  # one append == two appends
    assert np.array_equal(c.lat_codes, c2.lat_codes) and np.array_equal(c.idx_codes, c2.idx_codes)
    # one token per call, as a decode loop appends: the compression buffer carries the
    # odd token and the previous entry's b rows across calls; every plane and the
    # window ring end up as with one call
    c3 = orc.Cache(64, ratio=2)
    for j in range(n):
        orc.append_r2(c3, ca[j:j + 1], cb[j:j + 1], za[j:j + 1], zb[j:j + 1], ba, bb, 1e4)
    assert c3.n_tokens == 21 and c3.n_entries == 10
    for name in ("lat_codes", "lat_scales", "rope_codes", "rope_scales", "idx_codes", "idx_scales", "swa_codes",
                 "swa_scales"):
        assert np.array_equal(getattr(c3, name), getattr(c2, name)), name
    # [P5] §2.3.1: query t sees entries s < floor(t/m)
    assert orc.visible(20, 2) == 10 and orc.visible(21, 2) == 10 and orc.visible(19, 2) == 9
    # 8,192 tokens -> 4,096 entries (2 tokens per entry)
    assert 8192 // 2 == 4096
