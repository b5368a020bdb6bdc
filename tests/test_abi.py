"""Host-side checks of the C ABI (no GPU): the library builds, loads and exports
every function include/csa2.h declares; host validation returns the documented
status codes before any device work; the host RoPE table matches the oracle's."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fp4_compressed_sparse_gb300 import build_lib, csa2
    build_lib.build()
    return csa2.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    from fp4_compressed_sparse_gb300 import csa2
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(csa2.EXPORTS) == names


def test_status_strings_and_version(lib):
    assert lib.csa2_version() >= 100
    for s in range(8):
        assert lib.csa2_status_string(s)
    assert lib.csa2_status_string(99) == b"unknown status"


def test_host_validation_codes(lib):
    from fp4_compressed_sparse_gb300 import csa2
    # NULL cache
    assert lib.csa2_kv_append(None, None, None, 0, None, None, 1, 1, None, None, None) == 1
    assert b"cache" in lib.csa2_last_error_detail()
    # bad shapes / ranges before any device work (pointers are 16-aligned fakes, never touched)
    fake = 1 << 20
    st = csa2.CacheStruct(1, 16, 3, 1, *([fake] * 10))
    assert lib.csa2_kv_append(ctypes.byref(st), None, None, 0, None, None, 1, 1, None, None, None) == 4
    st = csa2.CacheStruct(0, 16, 1, 1, *([fake] * 10))
    assert lib.csa2_index_score(ctypes.byref(st), None, None, 4, None, None, 0, 8, None, 0, None, None, 0,
                                None, None) == 2
    st = csa2.CacheStruct(1, 16, 1, 1, *([fake] * 10))
    st.lat_codes = fake + 8  # misaligned
    assert lib.csa2_sparse_attn_decode(ctypes.byref(st), None, 64, None, None, 512, None, 0.1, None,
                                       None, None, 0, None, None) == 3
    st.lat_codes = fake
    p = ctypes.c_void_p(fake)
    # heads not a multiple of 16
    assert lib.csa2_sparse_attn_decode(ctypes.byref(st), p, 24, p, p, 512, None, 0.1, p, p, p, 1 << 20,
                                       None, None) == 2
    # k out of range
    assert lib.csa2_topk(p, 100, None, 1, 1, p, None, 0, 8, 0, p, 0, None, None, p, 1 << 20, None, None) == 4
    # workspace too small
    assert lib.csa2_topk(p, 100, None, 1, 1, p, None, 0, 8, 8, p, 0, None, None, p, 16, None, None) == 7
    # the candidate pool: at most 2048 blocks, built from 8-position blocks
    assert lib.csa2_topk(p, 100, None, 1, 1, p, None, 0, 8, 8, p, 4096, p, p, p, 1 << 20, None, None) == 4
    assert lib.csa2_topk(p, 100, None, 1, 1, p, None, 0, 16, 8, p, 64, p, p, p, 1 << 20, None, None) == 5
    # a misaligned sideband
    assert lib.csa2_topk(p, 100, ctypes.c_void_p(fake + 4), 1, 1, p, None, 0, 8, 8, p, 0, None, None, p,
                         1 << 20, None, None) == 3
    # prefill needs a ratio-2 cache
    assert lib.csa2_prefill_chunk(ctypes.byref(st), 0, None, p, 10, 4, p, p, 4, p, 16, 8, None, 0.1,
                                  p, p, p, p, 1 << 30, None, None) == 5


def test_rope_table_matches_oracle(lib, orc):
    n = 300
    host = np.zeros((n, 64), np.float32)
    assert lib.csa2_rope_table(10000.0, n, host.ctypes.data_as(ctypes.c_void_p)) == 0
    for pos in (0, 1, 17, 255, 299):
        assert np.array_equal(host[pos], orc.rope_cs(10000.0, pos))
    big = np.zeros((1, 64), np.float32)
    # a far position through the table formula (pos * theta^(-2i/64) in double)
    far = np.zeros((1048577, 64), np.float32)
    assert lib.csa2_rope_table(10000.0, far.shape[0], far.ctypes.data_as(ctypes.c_void_p)) == 0
    assert np.array_equal(far[1048576], orc.rope_cs(10000.0, 1048576))
    del big


def test_cache_plane_bytes_match_record(lib):
    # 288 B main + 36 B sidecar + 68 B indexer per entry; MXFP8 window 576 + scales
    per = [lib.csa2_cache_plane_bytes(1, 128, p, 1) / 128 for p in range(6)]
    assert per[0] + per[1] == 288 and per[2] + per[3] == 36 and per[4] + per[5] == 68
    # indexer planes are stored in whole 128-entry tiles
    assert lib.csa2_cache_plane_bytes(2, 129, 4, 1) == 2 * 2 * 8192
    assert lib.csa2_cache_plane_bytes(2, 129, 5, 1) == 2 * 2 * 512
    assert lib.csa2_cache_plane_bytes(1, 1, 6, 1) == 128 * 576
    assert lib.csa2_cache_plane_bytes(1, 1, 6, 0) == 128 * 1152


def test_topk_noalloc_failures_carry_their_own_detail(lib):
    """Every non-OK status of the no-allocation top-k sets its own detail text
    (a previous call's text must not leak through)."""
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    lib.csa2_topk_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    cases = [
        ((None, 100, 1, 1, fake, None, 0, 8, 16, fake, 0, None, None, None, None), 1, b"scores is NULL"),
        ((odd, 100, 1, 1, fake, None, 0, 8, 16, fake, 0, None, None, None, None), 3, b"scores is not 16-byte"),
        ((fake, 100, 0, 1, fake, None, 0, 8, 16, fake, 0, None, None, None, None), 2, b"batch 0"),
        ((fake, 100, 1, 3, fake, None, 0, 8, 16, fake, 0, None, None, None, None), 4, b"ratio 3"),
        ((fake, 100, 1, 1, fake, None, 0, 8, 0, fake, 0, None, None, None, None), 4, b"k 0"),
        ((fake, 100, 1, 1, fake, None, 0, 4, 16, fake, 64, fake, fake, None, None), 5, b"8-position"),
        ((fake, 1 << 26, 8, 1, fake, None, 0, 8, 16, fake, 0, None, None, None, None), 7, b"built-in array"),
    ]
    for args, status, text in cases:
        lib.csa2_set_phase_events(None, 0)  # an OK call in between: leaves the old detail behind
        assert lib.csa2_topk_noalloc(*args) == status, text
        assert text in lib.csa2_last_error_detail(), (text, lib.csa2_last_error_detail())


def test_measurement_helpers_validate(lib):
    assert lib.csa2_mxf4_peak_launch(0, 100, None, None, None) == 2
    assert lib.csa2_mxf4_peak_launch(152, 1, None, None, None) == 2
    assert b"iters" in lib.csa2_last_error_detail()
    assert lib.csa2_set_phase_events(None, 3) == 1
    fake = ctypes.c_void_p(1 << 20)
    assert lib.csa2_bounded_wait_check(0, 0, fake, None) == 2
    assert lib.csa2_bounded_wait_check(65, 0, fake, None) == 2
    assert lib.csa2_bounded_wait_check(4, 2, fake, None) == 4
    assert lib.csa2_bounded_wait_check(4, 0, None, None) == 1
    assert lib.csa2_bounded_wait_check(4, 0, ctypes.c_void_p((1 << 20) + 2), None) == 3
    assert b"4-byte" in lib.csa2_last_error_detail()
    assert lib.csa2_set_phase_events(None, 0) == 0 and lib.csa2_phase_events_recorded() == 0


def test_mask_to_pool_validates(lib):
    fake = ctypes.c_void_p(1 << 20)
    assert lib.csa2_mask_to_pool(None, 100, 1, 1, fake, fake, 8, 8, None) == 1
    assert lib.csa2_mask_to_pool(fake, 100, 1, 3, fake, fake, 8, 8, None) == 4
    assert lib.csa2_mask_to_pool(fake, 100, 1, 1, fake, fake, 8, 0, None) == 2
    assert b"pool_block_size" in lib.csa2_last_error_detail()


def test_paged_cache_validation(lib):
    from fp4_compressed_sparse_gb300 import csa2
    fake = 1 << 20
    st = csa2.CacheStruct(1, 512, 1, 1, *([fake] * 10), fake, 100, 5, 8, 0)  # page not a multiple of 128
    assert lib.csa2_index_score(ctypes.byref(st), None, None, 4, None, None, 0, 8, None, 0, None, None, 0,
                                None, None) == 2
    assert b"page_entries" in lib.csa2_last_error_detail()
    st = csa2.CacheStruct(1, 512, 1, 1, *([fake] * 10), fake, 128, 3, 8, 0)  # capacity != 3 x 128
    assert lib.csa2_kv_append(ctypes.byref(st), None, None, 0, None, None, 1, 1, None, None, None) == 2
    assert b"max_pages" in lib.csa2_last_error_detail()
    assert lib.csa2_paged_plane_bytes(10, 256, 0) == 10 * 256 * 256
    assert lib.csa2_paged_plane_bytes(10, 256, 4) == 10 * 2 * 8192
    assert lib.csa2_paged_plane_bytes(10, 100, 0) == 0
