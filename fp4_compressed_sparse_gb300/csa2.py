"""Thin Python binding of libcsa2 (ctypes).

Argument marshalling only: every step runs in libcsa2's CUDA kernels.  PyTorch
supplies device memory (caller-owned buffers) and the current CUDA stream.
There is no CPU fallback: if libcsa2.so is not built, load() raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build_lib

OK = 0
ERR_NAMES = {0: "OK", 1: "ERR_NULL", 2: "ERR_SHAPE", 3: "ERR_ALIGN", 4: "ERR_RANGE",
             5: "ERR_UNSUPPORTED", 6: "ERR_CUDA", 7: "ERR_WORKSPACE"}
DEVERR_CAPACITY, DEVERR_INDEX, DEVERR_NAN, DEVERR_ROPE, DEVERR_TIMEOUT, DEVERR_INEXACT = 1, 2, 4, 8, 16, 32
SWA_BF16, SWA_MXFP8 = 0, 1
ENTRY_FP4, ENTRY_FP8 = 0, 1
IN_F32, IN_BF16 = 0, 1
D_LATENT, D_ROPE, D_QK, D_INDEX, D_CMP, WINDOW = 512, 64, 576, 128, 704, 128

EXPORTS = [
    "csa2_cache_plane_bytes", "csa2_paged_plane_bytes", "csa2_entry_plane_bytes", "csa2_rope_table", "csa2_kv_append", "csa2_index_score_workspace_size",
    "csa2_score_aux_size", "csa2_index_score",
    "csa2_topk_workspace_size", "csa2_topk", "csa2_topk_noalloc", "csa2_attn_workspace_size", "csa2_sparse_attn_decode",
    "csa2_prefill_workspace_size", "csa2_prefill_chunk", "csa2_mask_to_pool", "csa2_mxf4_peak_launch",
    "csa2_bounded_wait_check", "csa2_set_phase_events",
    "csa2_phase_events_recorded", "csa2_status_string", "csa2_last_error_detail", "csa2_version",
]


class Csa2Error(RuntimeError):
    def __init__(self, fn, status, detail):
        super().__init__(f"{fn} -> {ERR_NAMES.get(status, status)}: {detail}")
        self.status = status


class CacheStruct(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("capacity", ctypes.c_int32), ("ratio", ctypes.c_int32),
        ("swa_dtype", ctypes.c_int32),
        ("lat_codes", ctypes.c_void_p), ("lat_scales", ctypes.c_void_p),
        ("rope_codes", ctypes.c_void_p), ("rope_scales", ctypes.c_void_p),
        ("idx_codes", ctypes.c_void_p), ("idx_scales", ctypes.c_void_p),
        ("swa_codes", ctypes.c_void_p), ("swa_scales", ctypes.c_void_p),
        ("cmp_buf", ctypes.c_void_p), ("n_tokens", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("page_entries", ctypes.c_int32), ("max_pages", ctypes.c_int32),
        ("n_pages", ctypes.c_int32), ("entry_format", ctypes.c_int32),
    ]


class CompressIn(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("ca", "cb", "za", "zb", "ba", "bb")]


_lib = None


def lib_path() -> str:
    return build_lib.LIB


def load() -> ctypes.CDLL:
    """Load libcsa2.so (built in-tree by build_lib.build()); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = build_lib.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libcsa2.so is not built ({path}); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(path)
    vp, i32, i64, f32, f64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                  ctypes.c_double, ctypes.c_size_t)
    sig = {
        "csa2_cache_plane_bytes": (sz, [i32, i32, i32, i32]),
        "csa2_paged_plane_bytes": (sz, [i32, i32, i32]),
        "csa2_entry_plane_bytes": (sz, [i32, i32]),
        "csa2_rope_table": (i32, [f64, i64, vp]),
        "csa2_kv_append": (i32, [vp, vp, vp, i32, vp, vp, i64, i32, vp, vp, vp]),
        "csa2_index_score_workspace_size": (sz, [i32, i32]),
        "csa2_score_aux_size": (sz, [i32, i64]),
        "csa2_index_score": (i32, [vp, vp, vp, i32, vp, vp, i32, i32, vp, i64, vp, vp, sz, vp, vp]),
        "csa2_topk_workspace_size": (sz, [i32, i64, i32, i32]),
        "csa2_topk": (i32, [vp, i64, vp, i32, i32, vp, vp, i32, i32, i32, vp, i32, vp, vp, vp, sz, vp, vp]),
        "csa2_topk_noalloc": (i32, [vp, i64, i32, i32, vp, vp, i32, i32, i32, vp, i32, vp, vp, vp, vp]),
        "csa2_attn_workspace_size": (sz, [i32, i32, i32]),
        "csa2_sparse_attn_decode": (i32, [vp, vp, i32, vp, vp, i32, vp, f32, vp, vp, vp, sz, vp, vp]),
        "csa2_prefill_workspace_size": (sz, [i32, i32, i32, i32, i32]),
        "csa2_prefill_chunk": (i32, [vp, i32, vp, vp, i64, i32, vp, vp, i32, vp, i32, i32, vp, f32,
                                     vp, vp, vp, vp, sz, vp, vp]),
        "csa2_mask_to_pool": (i32, [vp, i64, i32, i32, vp, vp, i32, i32, vp]),
        "csa2_mxf4_peak_launch": (i32, [i32, i32, vp, vp, vp]),
        "csa2_bounded_wait_check": (i32, [i32, i32, vp, vp]),
        "csa2_set_phase_events": (i32, [vp, i32]),
        "csa2_phase_events_recorded": (i32, []),
        "csa2_status_string": (ctypes.c_char_p, [i32]),
        "csa2_last_error_detail": (ctypes.c_char_p, []),
        "csa2_version": (i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(fn, status):
    if status != OK:
        detail = load().csa2_last_error_detail()
        raise Csa2Error(fn, status, detail.decode() if detail else "")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# --------------------------------------------------------------------------- cache
class Cache:
    """Caller-owned device planes of one global-KV cache (see csa2_cache in csa2.h).

    Dense by default: every entry plane is [batch][capacity][...].  With
    page_entries (a multiple of 128) the entry planes are a pool of n_pages
    physical pages of page_entries entries, and block_table [batch][max_pages]
    (int32, max_pages = capacity / page_entries) names the page that holds
    entries p*page_entries .. of each sequence; by default n_pages = batch *
    max_pages and the table is the identity."""

    def __init__(self, batch, capacity, ratio=1, swa_dtype=SWA_MXFP8, device="cuda", page_entries=None,
                 n_pages=None, block_table=None, entry_format=ENTRY_FP4):
        L = load()
        self.batch, self.capacity, self.ratio, self.swa_dtype = batch, capacity, ratio, swa_dtype
        self.page_entries, self.entry_format = page_entries, entry_format
        nb = [L.csa2_cache_plane_bytes(batch, capacity, p, swa_dtype) for p in range(10)]
        eb = [L.csa2_entry_plane_bytes(entry_format, p) for p in range(4)]  # bytes per entry, planes 0..3
        u8 = lambda n: torch.zeros(max(n, 16), dtype=torch.uint8, device=device)[:n]
        if page_entries:
            assert capacity % page_entries == 0 and page_entries % 128 == 0
            self.max_pages = capacity // page_entries
            self.n_pages = n_pages or batch * self.max_pages
            if block_table is None:
                block_table = torch.arange(batch * self.max_pages, dtype=torch.int32).view(batch, self.max_pages)
            self.block_table = block_table.to(device=device, dtype=torch.int32).contiguous()
            pb = [L.csa2_paged_plane_bytes(self.n_pages, page_entries, p) for p in range(6)]
            rows = self.n_pages * page_entries
            self.idx_tiles = rows // 128
            planes = [u8(rows * eb[p]).view(rows, eb[p]) if eb[p] else None for p in range(4)] + \
                     [u8(pb[4]).view(self.idx_tiles, 8192), u8(pb[5]).view(self.idx_tiles, 512)]
        else:
            self.max_pages = self.n_pages = 0
            self.block_table = None
            # tile-major indexer planes (see csa2_cache in csa2.h)
            self.idx_tiles = (capacity + 127) // 128
            n = batch * capacity
            planes = [u8(n * eb[p]).view(batch, capacity, eb[p]) if eb[p] else None for p in range(4)] + \
                     [u8(nb[4]).view(batch, self.idx_tiles, 8192), u8(nb[5]).view(batch, self.idx_tiles, 512)]
        (self.lat_codes, self.lat_scales, self.rope_codes, self.rope_scales, self.idx_codes,
         self.idx_scales) = planes
        sw = 576 if swa_dtype == SWA_MXFP8 else 1152
        self.swa_codes = u8(nb[6]).view(batch, WINDOW, sw)
        self.swa_scales = u8(nb[7]).view(batch, WINDOW, 32)
        self.cmp_buf = torch.zeros(batch, 4, 4, D_CMP, dtype=torch.float32, device=device) \
            if ratio == 2 else None
        self.n_tokens = torch.zeros(batch, dtype=torch.int64, device=device)
        self.struct = CacheStruct(
            batch, capacity, ratio, swa_dtype,
            self.lat_codes.data_ptr(), self.lat_scales.data_ptr(), self.rope_codes.data_ptr(),
            self.rope_scales.data_ptr() if self.rope_scales is not None else None, self.idx_codes.data_ptr(),
            self.idx_scales.data_ptr(), self.swa_codes.data_ptr(), self.swa_scales.data_ptr(),
            self.cmp_buf.data_ptr() if self.cmp_buf is not None else None, self.n_tokens.data_ptr(),
            self.block_table.data_ptr() if self.block_table is not None else None, page_entries or 0,
            self.max_pages, self.n_pages, entry_format)

    def ref(self):
        return ctypes.byref(self.struct)

    def _rows(self):
        """Physical entry row of every (sequence, entry) of a paged cache: [B, cap] int64."""
        pe = self.page_entries
        pages = self.block_table.to(torch.int64)  # [B, max_pages]
        return (pages[:, :, None] * pe + torch.arange(pe, device=pages.device)).reshape(self.batch, -1)

    def plane(self, name):
        """Entry plane `name` (lat_codes, lat_scales, rope_codes, rope_scales) per sequence: [B, cap, bytes]."""
        t = getattr(self, name)
        return t if not self.page_entries else t[self._rows()]

    def idx_entries(self):
        """The indexer planes re-read per entry: (codes [B,cap,64], scales [B,cap,4])."""
        if self.page_entries:
            nt = self.idx_tiles
            codes = self.idx_codes.view(nt, 4, 128, 16).permute(0, 2, 1, 3).reshape(nt * 128, 64)
            scales = self.idx_scales.view(nt, 32, 4, 4).permute(0, 2, 1, 3).reshape(nt * 128, 4)
            rows = self._rows()
            return codes[rows], scales[rows]
        B, nt = self.batch, self.idx_tiles
        codes = self.idx_codes.view(B, nt, 4, 128, 16).permute(0, 1, 3, 2, 4).reshape(B, nt * 128, 64)
        scales = self.idx_scales.view(B, nt, 32, 4, 4).permute(0, 1, 3, 2, 4).reshape(B, nt * 128, 4)
        return codes[:, :self.capacity], scales[:, :self.capacity]

    def entry_bytes(self):
        """Bytes of one stored entry: main record + RoPE part + indexer key (68): 288 + 36 + 68
        for the V4.1 FP4 format, 528 + 128 + 68 for the V4 format."""
        L = load()
        return sum(L.csa2_entry_plane_bytes(self.entry_format, p) for p in range(6))


def rope_table(theta: float, n_pos: int, device="cuda") -> torch.Tensor:
    """csa2_rope_table (host) copied to the device: [n_pos, 32, 2] fp32."""
    host = torch.empty((n_pos, 32, 2), dtype=torch.float32)
    _check("csa2_rope_table", load().csa2_rope_table(float(theta), int(n_pos),
                                                     ctypes.c_void_p(host.data_ptr())))
    return host.to(device)


def kv_append(cache: Cache, kv=None, idx_key=None, rope_cs=None, cmp=None, cmp_dbg=None,
              err=None, stream=None):
    """csa2_kv_append.  Ratio 1: kv [B,n,576], idx_key [B,n,128] (fp32 or bf16).
    Ratio 2: cmp = (ca, cb, za, zb [B,n,704], ba, bb [2,704]) fp32."""
    L = load()
    if cache.ratio == 1:
        n_new = kv.shape[1]
        dt = IN_BF16 if kv.dtype == torch.bfloat16 else IN_F32
        cin = None
    else:
        n_new = cmp[0].shape[1]
        dt = IN_F32
        cin = CompressIn(*[t.data_ptr() for t in cmp])
    st = L.csa2_kv_append(cache.ref(), _ptr(kv), _ptr(idx_key), dt,
                          ctypes.byref(cin) if cin is not None else None, _ptr(rope_cs),
                          rope_cs.shape[0], n_new, _ptr(cmp_dbg), _ptr(err), _stream(stream))
    _check("csa2_kv_append", st)


def index_score_workspace(batch, heads_idx, device="cuda"):
    n = load().csa2_index_score_workspace_size(batch, heads_idx)
    return torch.empty(n, dtype=torch.uint8, device=device)


def score_aux(batch, stride, device="cuda"):
    """A buffer for the score sideband csa2_index_score can leave for csa2_topk."""
    n = load().csa2_score_aux_size(batch, stride)
    return torch.empty(n, dtype=torch.uint8, device=device)


_ws_cache = {}


def index_score(cache: Cache, q_idx, w, q_pos, scores, pool=None, pool_block_size=8, err=None,
                stream=None, ws=None, aux=None):
    """csa2_index_score: q_idx bf16 [B,H_I,128], w fp32 [B,H_I], q_pos int64 [B],
    scores fp32 [B, stride]; pool int32 [B, pool_blocks] for a Reindex layer;
    aux (optional, from score_aux()) receives the sideband for topk()."""
    L = load()
    if ws is None:
        key = (q_idx.shape[0], q_idx.shape[1], q_idx.device)
        ws = _ws_cache.get(key)
        if ws is None:
            ws = _ws_cache[key] = index_score_workspace(q_idx.shape[0], q_idx.shape[1], q_idx.device)
    st = L.csa2_index_score(cache.ref(), _ptr(q_idx), _ptr(w), q_idx.shape[1], _ptr(q_pos),
                            _ptr(pool), pool.shape[1] if pool is not None else 0, pool_block_size,
                            _ptr(scores), scores.shape[1], _ptr(aux), _ptr(ws), ws.numel(), _ptr(err),
                            _stream(stream))
    _check("csa2_index_score", st)


def topk_workspace(batch, stride, k, out_pool_blocks=0, device="cuda"):
    n = load().csa2_topk_workspace_size(batch, stride, k, out_pool_blocks)
    return torch.empty(n, dtype=torch.uint8, device=device)


def topk(scores, ratio, q_pos, k, idx_out, ws, pool=None, pool_block_size=8, pool_out=None,
         pool_count=None, err=None, stream=None, aux=None):
    """csa2_topk over the candidates csa2_index_score scored (aux: its sideband, or None)."""
    L = load()
    st = L.csa2_topk(_ptr(scores), scores.shape[1], _ptr(aux), scores.shape[0], ratio, _ptr(q_pos), _ptr(pool),
                     pool.shape[1] if pool is not None else 0, pool_block_size, k, _ptr(idx_out),
                     pool_out.shape[1] if pool_out is not None else 0, _ptr(pool_out), _ptr(pool_count),
                     _ptr(ws), ws.numel(), _ptr(err), _stream(stream))
    _check("csa2_topk", st)


def topk_noalloc(scores, ratio, q_pos, k, idx_out, pool=None, pool_block_size=8, pool_out=None,
                 pool_count=None, err=None, stream=None):
    """csa2_topk_noalloc: csa2_topk with the library's built-in 4 MiB scratch instead of a
    caller workspace (for callers that cannot allocate device memory while running)."""
    L = load()
    st = L.csa2_topk_noalloc(_ptr(scores), scores.shape[1], scores.shape[0], ratio, _ptr(q_pos),
                             _ptr(pool), pool.shape[1] if pool is not None else 0, pool_block_size, k,
                             _ptr(idx_out), pool_out.shape[1] if pool_out is not None else 0,
                             _ptr(pool_out), _ptr(pool_count), _ptr(err), _stream(stream))
    _check("csa2_topk_noalloc", st)


def attn_workspace(batch, heads, k, device="cuda"):
    n = load().csa2_attn_workspace_size(batch, heads, k)
    return torch.empty(n, dtype=torch.uint8, device=device)


def sparse_attn_decode(cache: Cache, q, q_pos, idx, out, lse, ws, sm_scale, sink=None, err=None,
                       stream=None):
    """csa2_sparse_attn_decode: q bf16 [B,H,576], idx int32 [B,k] -> out [B,H,512], lse [B,H]."""
    L = load()
    st = L.csa2_sparse_attn_decode(cache.ref(), _ptr(q), q.shape[1], _ptr(q_pos), _ptr(idx),
                                   idx.shape[1], _ptr(sink), float(sm_scale), _ptr(out), _ptr(lse),
                                   _ptr(ws), ws.numel(), _ptr(err), _stream(stream))
    _check("csa2_sparse_attn_decode", st)


def prefill_workspace(Q, capacity, heads_idx, heads, k, device="cuda"):
    n = load().csa2_prefill_workspace_size(Q, capacity, heads_idx, heads, k)
    return torch.empty(n, dtype=torch.uint8, device=device)


def prefill_chunk(cache: Cache, seq, cmp, rope_cs, q_idx, w, q, k, sm_scale, idx_out, out, lse, ws,
                  sink=None, err=None, stream=None):
    """csa2_prefill_chunk for sequence `seq` of a ratio-2 cache."""
    L = load()
    cin = CompressIn(*[t.data_ptr() for t in cmp])
    Q = cmp[0].shape[-2]
    st = L.csa2_prefill_chunk(cache.ref(), seq, ctypes.byref(cin), _ptr(rope_cs), rope_cs.shape[0], Q,
                              _ptr(q_idx), _ptr(w), q_idx.shape[1], _ptr(q), q.shape[1], k, _ptr(sink),
                              float(sm_scale), _ptr(idx_out), _ptr(out), _ptr(lse), _ptr(ws),
                              ws.numel(), _ptr(err), _stream(stream))
    _check("csa2_prefill_chunk", st)


def mask_to_pool(scores, ratio, q_pos, pool, pool_block_size=8, stream=None):
    """Set FULL-mode scores outside each row's candidate pool to -inf, in place
    (the Reindex form of the published reference code)."""
    B, stride = scores.shape
    _check("csa2_mask_to_pool", load().csa2_mask_to_pool(_ptr(scores), stride, B, ratio, _ptr(q_pos), _ptr(pool),
                                                          pool.shape[1], pool_block_size, _stream(stream)))


# --------------------------------------------------------------------------- measurement helpers
def mxf4_peak_launch(n_ctas, iters, sink=None, err=None, stream=None):
    """Back-to-back block-scaled FP4 MMAs (M 128 x N 128 x K 64) on every CTA;
    the caller times it: n_ctas * iters * 2 * 128 * 128 * 64 FLOP."""
    _check("csa2_mxf4_peak_launch", load().csa2_mxf4_peak_launch(n_ctas, iters, _ptr(sink), _ptr(err),
                                                                  _stream(stream)))


def bounded_wait_check(iters, complete, err, stream=None):
    """One warp holding tensor memory across the library's bounded mbarrier wait:
    complete=True -> the wait succeeds; False -> it gives up after `iters` polls
    (<= ~1 ms each) and ORs DEVERR_TIMEOUT into `err` (int32 device tensor)."""
    _check("csa2_bounded_wait_check", load().csa2_bounded_wait_check(iters, 1 if complete else 0, _ptr(err),
                                                                      _stream(stream)))


_phase_keep = None


def set_phase_events(events):
    """Record the given torch.cuda.Events at the phase boundaries of this thread's
    next prefill_chunk calls (None or [] stops); each must have been recorded once
    so that its CUDA event exists."""
    global _phase_keep
    if not events:
        _phase_keep = None
        _check("csa2_set_phase_events", load().csa2_set_phase_events(None, 0))
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _phase_keep = arr
    _check("csa2_set_phase_events", load().csa2_set_phase_events(arr, len(events)))


def phase_events_recorded():
    return int(load().csa2_phase_events_recorded())
