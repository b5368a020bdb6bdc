"""CPU oracle for the CSA2 long-context attention step -- Python side.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference arm of bench.py may import this module.  The product
path (libcsa2 and its binding) never imports it and shares no code with it.

The arithmetic lives in ``csa2_oracle.c`` (plain C, fp64 where the pages fix
no precision, compiled with -fno-fast-math -ffp-contract=off).  This module
only marshals numpy arrays and strings together the per-step functions in the
order the pages give them:

  append (quantise after RoPE) -> index score -> top-k (+ candidate pool)
  -> sparse attention over the selected entries plus the sliding window.

Page names used in the citations:
  [P1] "DeepSeek V4.1 Flash 아키텍처 분석" (plaidlabs.ai blog)
  [P2] "DeepSeek Multi-Head Latent Attention(MLA) 해부" (huny.dev blog)
  [P3] "DeepSeek V4.1 Flash 해부, KV 캐시는 줄고 사후학습 레시피는 그대로" (traillabs.ai)
  [P4] "매개변수는 커졌는데 메모리는 4분의 1, DeepSeek V4.1 Flash의 KV 캐시 다이어트" (ithotfix.com)
  [P5] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence" (issue #58 translation)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

LAT = 512   # latent dims ([P1] "890 bytes/token")
ROPE = 64   # decoupled RoPE dims ([P2] §3)
DQK = 576   # LAT + ROPE
DI = 128    # indexer head dim c_I ([P5] §4.2.1)
WIN = 128   # sliding window n_win ([P5] §4.2.1)

SWA_BF16 = 0
SWA_MXFP8 = 1


def build(force: bool = False) -> str:
    """Compile csa2_oracle.c into oracle/_build/liboracle.so (atomic rename)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _declare(L):
    vp, i32, i64, f32, f64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                              ctypes.c_float, ctypes.c_double)
    u8, u16 = ctypes.c_uint8, ctypes.c_uint16
    sig = {
        "orc_e2m1_decode": (f64, [u8]),
        "orc_e2m1_encode": (u8, [f32]),
        "orc_e4m3_decode": (f64, [u8]),
        "orc_e4m3_encode": (u8, [f32]),
        "orc_e8m0_decode": (f64, [u8]),
        "orc_bf16_encode": (u16, [f32]),
        "orc_bf16_decode": (f64, [u16]),
        "orc_nvfp4_quant16": (None, [vp, vp, vp]),
        "orc_mxfp4_quant32": (None, [vp, vp, vp]),
        "orc_mxfp8_quant32": (None, [vp, vp, vp]),
        "orc_rope_cs": (None, [f64, i64, vp]),
        "orc_rope_apply": (None, [vp, vp]),
        "orc_encode_entry": (None, [vp] * 9),
        "orc_encode_entry_v4": (None, [vp] * 8),
        "orc_encode_swa": (None, [vp, vp, i32, vp, vp]),
        "orc_encode_keys": (None, [i64, vp, vp, vp]),
        "orc_compress": (None, [i32, i32, vp, vp, vp, vp, vp, vp, vp]),
        "orc_quant_q_index": (None, [i32, vp, vp, vp]),
        "orc_index_score_rows": (i32, [i64, vp, vp, vp, i32, vp, vp, vp]),
        "orc_topk": (i32, [i64, vp, vp, i32, vp]),
        "orc_pool": (i32, [i64, vp, i32, i32, vp, vp]),
        "orc_dequant_main": (None, [vp, vp, vp, vp, vp]),
        "orc_dequant_swa": (None, [vp, vp, i32, vp]),
        "orc_sparse_attn": (i32, [i32, vp, vp, vp, vp, vp, vp, i32, vp, i64, vp, i64, i32, i32,
                                  vp, f32, vp, vp, i32]),
        "orc_main_entry_bytes": (i32, [i32, i32]),
        "orc_mx_entry_bytes": (i32, [i32, i32]),
        "orc_num_threads": (i32, []),
        "orc_set_num_threads": (None, [i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops over independent rows from now on."""
    lib().orc_set_num_threads(int(n))


# --------------------------------------------------------------------------
# Formats (C1) and group quantisers (C3)
# --------------------------------------------------------------------------
def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(code)


def e2m1_encode(x: float) -> int:
    return lib().orc_e2m1_encode(x)


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(code)


def e4m3_encode(x: float) -> int:
    return lib().orc_e4m3_encode(x)


def e8m0_decode(code: int) -> float:
    return lib().orc_e8m0_decode(code)


def bf16_encode(x: float) -> int:
    return lib().orc_bf16_encode(x)


def bf16_decode(h: int) -> float:
    return lib().orc_bf16_decode(h)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def nvfp4_quant16(x):
    """One group of 16 values -> (8 packed code bytes, E4M3 scale byte)."""
    x = _f32(x)
    assert x.shape == (16,)
    codes = np.zeros(8, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib().orc_nvfp4_quant16(_p(x), _p(codes), _p(sc))
    return codes, int(sc[0])


def mxfp4_quant32(x):
    x = _f32(x)
    assert x.shape == (32,)
    codes = np.zeros(16, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib().orc_mxfp4_quant32(_p(x), _p(codes), _p(sc))
    return codes, int(sc[0])


def mxfp8_quant32(x):
    x = _f32(x)
    assert x.shape == (32,)
    codes = np.zeros(32, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib().orc_mxfp8_quant32(_p(x), _p(codes), _p(sc))
    return codes, int(sc[0])


def unpack_fp4(codes: np.ndarray) -> np.ndarray:
    """Packed bytes [..., n/2] -> 4-bit codes [..., n] (low nibble first)."""
    codes = np.asarray(codes, np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = codes & 15
    out[..., 1::2] = codes >> 4
    return out


def dequant_nvfp4(codes, scales):
    """[..., n/2] codes + [..., n/16] E4M3 scales -> fp64 [..., n]."""
    c = unpack_fp4(codes)
    mag = np.array([lib().orc_e2m1_decode(i) for i in range(16)])
    sc = np.array([lib().orc_e4m3_decode(i) for i in range(256)])
    v = mag[c]
    s = np.repeat(sc[np.asarray(scales, np.uint8)], 16, axis=-1)
    return v * s


def dequant_mxfp4(codes, scales):
    c = unpack_fp4(codes)
    mag = np.array([lib().orc_e2m1_decode(i) for i in range(16)])
    sc = np.array([lib().orc_e8m0_decode(i) for i in range(256)])
    return mag[c] * np.repeat(sc[np.asarray(scales, np.uint8)], 32, axis=-1)


# --------------------------------------------------------------------------
# RoPE (C9)
# --------------------------------------------------------------------------
def rope_cs(theta: float, pos: int) -> np.ndarray:
    cs = np.zeros(64, np.float32)
    lib().orc_rope_cs(float(theta), int(pos), _p(cs))
    return cs


def rope_apply(x64, cs):
    x = _f32(x64).copy()
    lib().orc_rope_apply(_p(x), _p(_f32(cs)))
    return x


# --------------------------------------------------------------------------
# Cache built by the oracle (host numpy arrays, one sequence)
# --------------------------------------------------------------------------
# Main-entry formats: bytes per entry of (lat_codes, lat_scales, rope_codes, rope_scales)
ENTRY_FP4, ENTRY_FP8 = 0, 1
ENTRY_PLANES = {
    ENTRY_FP4: (256, 32, 32, 4),   # V4.1: the 288 B record + the 36 B RoPE sidecar
    ENTRY_FP8: (512, 16, 128, 1),  # V4 ([P5] §2.3.4): E4M3 + E8M0 per 32 (528 B), RoPE in bf16 (128 B)
}


class Cache:
    """One sequence's cache, laid out like the pages' records.

    lat_codes [cap,256] lat_scales [cap,32]   -> 288 B main entry ([P1] "890 bytes/token")
    rope_codes [cap,32] rope_scales [cap,4]   -> 36 B RoPE sidecar (READING: MLA split, [P2] §3)
    idx_codes [cap,64]  idx_scales [cap,4]    -> 68 B MXFP4 indexer key
    swa_codes [WIN, 576 or 1152] swa_scales [WIN, 18] -> window ring, slot = token % WIN
    """

    def __init__(self, cap: int, swa_dtype: int = SWA_MXFP8, ratio: int = 1, entry_format: int = ENTRY_FP4):
        self.cap = cap
        self.ratio = ratio
        self.swa_dtype = swa_dtype
        self.entry_format = entry_format
        lat, lsc, rop, rsc = ENTRY_PLANES[entry_format]
        self.lat_codes = np.zeros((cap, lat), np.uint8)
        self.lat_scales = np.zeros((cap, lsc), np.uint8)
        self.rope_codes = np.zeros((cap, rop), np.uint8)
        self.rope_scales = np.zeros((cap, rsc), np.uint8)
        self.idx_codes = np.zeros((cap, 64), np.uint8)
        self.idx_scales = np.zeros((cap, 4), np.uint8)
        sw = 576 if swa_dtype == SWA_MXFP8 else 1152
        self.swa_codes = np.zeros((WIN, sw), np.uint8)
        self.swa_scales = np.zeros((WIN, 18), np.uint8)
        self.n_tokens = 0
        self.n_entries = 0
        # ratio-2 compression inputs of every token so far (the oracle keeps them all)
        self._cmp_rows = []


def encode_entry(v576, ik128, cs):
    """fp32 entry vector (rope dims unrotated) + indexer key -> the record bytes."""
    v, ik = _f32(v576), _f32(ik128)
    out = [np.zeros(n, np.uint8) for n in (256, 32, 32, 4, 64, 4)]
    lib().orc_encode_entry(_p(v), _p(ik), _p(_f32(cs)), *[_p(o) for o in out])
    return out


class KeyCache:
    """Indexer-key records only (what the index score reads): idx_codes [n,64],
    idx_scales [n,4] of n consecutive entries."""

    def __init__(self, n: int):
        self.idx_codes = np.zeros((n, 64), np.uint8)
        self.idx_scales = np.zeros((n, 4), np.uint8)


def encode_keys(cache, start: int, ik):
    """MXFP4 records of the indexer keys ik [n,128] into entries start.. of a
    KeyCache or Cache (the idx planes of encode_entry, [P5] §2.3.4)."""
    ik = _f32(ik)
    n = ik.shape[0]
    codes = np.zeros((n, 64), np.uint8)
    scales = np.zeros((n, 4), np.uint8)
    lib().orc_encode_keys(n, _p(ik), _p(codes), _p(scales))
    cache.idx_codes[start:start + n] = codes
    cache.idx_scales[start:start + n] = scales


def encode_entry_v4(v576, ik128, cs):
    """The V4 entry ([P5] §2.3.4: FP8 except the RoPE dims, kept bf16): the record
    bytes (lat_codes 512, lat_scales 16, rope_codes 128, rope_scales (unused) 1,
    idx_codes 64, idx_scales 4)."""
    v, ik = _f32(v576), _f32(ik128)
    out = [np.zeros(n, np.uint8) for n in (512, 16, 128, 1, 64, 4)]
    lib().orc_encode_entry_v4(_p(v), _p(ik), _p(_f32(cs)), _p(out[0]), _p(out[1]), _p(out[2]), _p(out[4]),
                              _p(out[5]))
    return out


def encode_for(cache, v576, ik128, cs):
    """The record of an entry in the cache's entry format."""
    if getattr(cache, "entry_format", ENTRY_FP4) == ENTRY_FP8:
        return encode_entry_v4(v576, ik128, cs)
    return encode_entry(v576, ik128, cs)


def encode_swa(v576, cs, swa_dtype):
    codes = np.zeros(576 if swa_dtype == SWA_MXFP8 else 1152, np.uint8)
    scales = np.zeros(18, np.uint8)
    lib().orc_encode_swa(_p(_f32(v576)), _p(_f32(cs)), int(swa_dtype == SWA_MXFP8), _p(codes),
                         _p(scales))
    return codes, scales


def append_r1(cache: Cache, kv, ik, theta: float):
    """Decoder-style append (1 token = 1 entry): RoPE, then quantise ([P4] "890이
    맞아떨어지는 계산": quantisation after RoPE); the token also fills its window
    slot (token % WIN) in 8 bits ([P1] "890 bytes/token": window KV in FP8)."""
    kv, ik = _f32(kv), _f32(ik)
    n = kv.shape[0]
    assert cache.ratio == 1 and cache.n_tokens + n <= cache.cap
    for j in range(n):
        t = cache.n_tokens + j
        cs = rope_cs(theta, t)
        rec = encode_for(cache, kv[j], ik[j], cs)
        for arr, val in zip((cache.lat_codes, cache.lat_scales, cache.rope_codes,
                             cache.rope_scales, cache.idx_codes, cache.idx_scales), rec):
            arr[t] = val
        if j >= n - WIN:
            c, s = encode_swa(kv[j], cs, cache.swa_dtype)
            cache.swa_codes[t % WIN] = c
            cache.swa_scales[t % WIN] = s
    cache.n_tokens += n
    cache.n_entries = cache.n_tokens


def compress_entry(m, ca_rows, za_rows, cb_rows, zb_rows, ba, bb):
    """C10: one compressed entry from m 'a' rows and m 'b' rows (b rows None for
    entry 0), each row [dim]; returns fp32 [dim]."""
    dim = ca_rows[0].shape[0]
    arr_t = ctypes.c_void_p * m
    keep = []

    def rows(lst):
        if lst is None:
            return None
        lst = [_f32(r) for r in lst]
        keep.extend(lst)
        return arr_t(*[r.ctypes.data for r in lst])

    out = np.zeros(dim, np.float32)
    ba, bb = _f32(ba), _f32(bb)
    lib().orc_compress(m, dim, rows(ca_rows), rows(za_rows), rows(cb_rows), rows(zb_rows),
                       _p(ba), _p(bb), _p(out))
    return out


def append_r2(cache: Cache, ca, cb, za, zb, ba, bb, theta: float, dbg=None):
    """Encoder-style append, 2 tokens per entry ([P5] §2.3.1 compression with
    m = 2; [P1]/[P4]: encoder caches pack 2 tokens into one entry).

    ca, cb, za, zb: [n, 704] per token (576 main dims then 128 indexer dims).
    ba, bb: [2, 704].  Entry i is emitted once tokens 2i, 2i+1 are present.
    READING: RoPE of entry i at position 2i (its first token); the window slot of
    token t holds its own C^a row, rotated at t.
    If dbg is a list, the fp32 compressed entries (before RoPE) are appended to it.
    """
    ca, cb, za, zb = (_f32(a) for a in (ca, cb, za, zb))
    n = ca.shape[0]
    assert cache.ratio == 2
    for j in range(n):
        cache._cmp_rows.append((ca[j], cb[j], za[j], zb[j]))
        t = cache.n_tokens + j
        if j >= n - WIN:
            cs = rope_cs(theta, t)
            c, s = encode_swa(ca[j, :576], cs, cache.swa_dtype)
            cache.swa_codes[t % WIN] = c
            cache.swa_scales[t % WIN] = s
    cache.n_tokens += n
    rows = cache._cmp_rows
    while 2 * cache.n_entries + 2 <= cache.n_tokens:
        i = cache.n_entries
        a = [rows[2 * i], rows[2 * i + 1]]
        b = [rows[2 * i - 2], rows[2 * i - 1]] if i > 0 else None
        v = compress_entry(2, [r[0] for r in a], [r[2] for r in a],
                           [r[1] for r in b] if b else None, [r[3] for r in b] if b else None,
                           ba, bb)
        if dbg is not None:
            dbg.append(v.copy())
        cs = rope_cs(theta, 2 * i)
        rec = encode_for(cache, v[:576], v[576:], cs)
        for arr, val in zip((cache.lat_codes, cache.lat_scales, cache.rope_codes,
                             cache.rope_scales, cache.idx_codes, cache.idx_scales), rec):
            arr[i] = val
        cache.n_entries += 1


# --------------------------------------------------------------------------
# Indexer (C4), top-k (C6), pool (C7)
# --------------------------------------------------------------------------
def visible(q_pos: int, ratio: int) -> int:
    """[P5] §2.3.1: entry s is visible to query t iff s < floor(t/m)."""
    return q_pos // ratio


def index_scores(cache: Cache, q_idx_bf16, w, n_vis=None, rows=None):
    """Scores of rows (or of positions 0..n_vis-1). q_idx_bf16: uint16 [H_I,128]."""
    q = np.ascontiguousarray(q_idx_bf16, np.uint16)
    w = _f32(w)
    H = q.shape[0]
    if rows is not None:
        rows = np.ascontiguousarray(rows, np.int64)
        n = rows.shape[0]
    else:
        n = int(n_vis)
    out = np.zeros(n, np.float32)
    flags = lib().orc_index_score_rows(n, _p(cache.idx_codes), _p(cache.idx_scales),
                                       _p(rows) if rows is not None else None, H, _p(q), _p(w),
                                       _p(out))
    return out, int(flags)


def topk(scores, k, positions=None):
    s = _f32(scores)
    pos = None if positions is None else np.ascontiguousarray(positions, np.int64)
    out = np.zeros(k, np.int32)
    rc = lib().orc_topk(s.shape[0], _p(s), _p(pos) if pos is not None else None, k, _p(out))
    if rc != 0:
        raise ValueError("NaN score")
    return out


def pool(scores, T, block_size=8, max_blocks=2048):
    s = _f32(scores)
    out = np.zeros(max_blocks, np.int32)
    cnt = np.zeros(1, np.int32)
    rc = lib().orc_pool(int(T), _p(s), block_size, max_blocks, _p(out), _p(cnt))
    if rc != 0:
        raise ValueError("NaN score")
    return out, int(cnt[0])


def pool_positions(pool_ids, count, T, block_size=8):
    """Visible positions inside the pool blocks, ascending."""
    ids = np.asarray(pool_ids[:count], np.int64)
    pos = (ids[:, None] * block_size + np.arange(block_size)[None, :]).reshape(-1)
    return pos[pos < T]


# --------------------------------------------------------------------------
# Sparse attention (C8)
# --------------------------------------------------------------------------
def swa_tokens(q_pos: int, n_tokens: int):
    """Window tokens of the query at q_pos: max(0, q_pos-127) .. q_pos."""
    lo = max(0, q_pos - WIN + 1)
    hi = min(q_pos, n_tokens - 1)
    return list(range(lo, hi + 1))


def sparse_attn(cache: Cache, q_bf16, idx, q_pos: int, sm_scale: float, sink=None,
                swa_codes=None, swa_scales=None):
    """q_bf16: uint16 [H,576]; idx: int32 [k] (-1 = empty).  The window rows are
    the cache ring slots of swa_tokens(q_pos) unless swa_codes/scales are given."""
    q = np.ascontiguousarray(q_bf16, np.uint16)
    H = q.shape[0]
    idx = np.ascontiguousarray(idx, np.int32)
    if swa_codes is None:
        toks = swa_tokens(q_pos, cache.n_tokens)
        slots = np.array([t % WIN for t in toks], np.int64)
        swa_codes = np.ascontiguousarray(cache.swa_codes[slots])
        swa_scales = np.ascontiguousarray(cache.swa_scales[slots])
    swa_codes = np.ascontiguousarray(swa_codes, np.uint8)
    swa_scales = np.ascontiguousarray(swa_scales, np.uint8)
    n_swa = swa_codes.shape[0]
    out = np.zeros((H, 512), np.float32)
    lse = np.zeros(H, np.float32)
    sk = None if sink is None else _f32(sink)
    lib().orc_sparse_attn(H, _p(q), _p(cache.lat_codes), _p(cache.lat_scales), _p(cache.rope_codes),
                          _p(cache.rope_scales), _p(idx), idx.shape[0], _p(swa_codes),
                          swa_codes.shape[1] if n_swa else 0, _p(swa_scales), 18, n_swa,
                          int(cache.swa_dtype == SWA_MXFP8), _p(sk) if sk is not None else None,
                          float(sm_scale), _p(out), _p(lse), int(getattr(cache, "entry_format", ENTRY_FP4)))
    return out, lse


# --------------------------------------------------------------------------
# Layer roles ([P3] "CSA2의 세 가지 모드"; [P4] "40개 층 중 바이트를 쓰는 곳은 넷")
# --------------------------------------------------------------------------
def full_layer(cache: Cache, q_idx, w, q, q_pos, k, sm_scale, sink=None, pool_blocks=2048,
               pool_block_size=8):
    """Full: score every visible entry, keep the top k, build the candidate pool,
    attend.  Returns (idx, pool_ids, pool_count, out, lse, scores)."""
    T = visible(q_pos, cache.ratio)
    scores, flags = index_scores(cache, q_idx, w, n_vis=T)
    assert flags == 0, f"index score exactness flags {flags}"
    idx = topk(scores, k)
    pids, cnt = pool(scores, T, pool_block_size, pool_blocks)
    out, lse = sparse_attn(cache, q, idx, q_pos, sm_scale, sink)
    return idx, pids, cnt, out, lse, scores


def reindex_layer(cache: Cache, q_idx, w, q, q_pos, k, sm_scale, pool_ids, pool_count, sink=None,
                  pool_block_size=8):
    """Reindex: score only the visible positions of the candidate pool, keep top k."""
    T = visible(q_pos, cache.ratio)
    pos = pool_positions(pool_ids, pool_count, T, pool_block_size)
    scores, flags = index_scores(cache, q_idx, w, rows=pos)
    assert flags == 0, f"index score exactness flags {flags}"
    idx = topk(scores, k, positions=pos)
    out, lse = sparse_attn(cache, q, idx, q_pos, sm_scale, sink)
    return idx, out, lse, scores, pos


def reuse_layer(cache: Cache, q, q_pos, idx, sm_scale, sink=None):
    """Reuse: the leader's KV and index list, this layer's own query; no indexer."""
    return sparse_attn(cache, q, idx, q_pos, sm_scale, sink)
