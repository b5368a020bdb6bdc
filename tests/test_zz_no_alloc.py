"""csa2_topk_noalloc: the top-k entry point for callers that may not allocate
device memory while running (its scratch is an array built into the library).
Checked through the C ABI against csa2_topk with a caller workspace, on two
calls in a row (the shared array keeps the previous call's contents)."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _scores(csa2, B, T, H_I, seed):
    c = csa2.Cache(B, T + 8, ratio=1)
    rope = csa2.rope_table(1e4, T + 16)
    g = torch.Generator(device="cuda").manual_seed(seed)
    kv = torch.randn((B, T, 576), generator=g, device="cuda")
    ik = torch.randn((B, T, 128), generator=g, device="cuda")
    csa2.kv_append(c, kv, ik, rope)
    q_idx = torch.randn((B, H_I, 128), generator=g, device="cuda").to(torch.bfloat16)
    w = torch.rand((B, H_I), generator=g, device="cuda")
    q_pos = torch.full((B,), T - 1, dtype=torch.int64, device="cuda")
    scores = torch.empty((B, c.capacity), device="cuda")
    csa2.index_score(c, q_idx, w, q_pos, scores)
    return c, scores, q_pos


def _call_noalloc(L, scores, q_pos, k, idx, pool_out=None, pool_cnt=None, pool=None):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.csa2_topk_noalloc(p(scores), scores.shape[1], scores.shape[0], 1, p(q_pos), p(pool),
                               pool.shape[1] if pool is not None else 0, 8, k, p(idx),
                               pool_out.shape[1] if pool_out is not None else 0, p(pool_out),
                               p(pool_cnt), None, stream)


def test_topk_noalloc_matches_workspace_version():
    from fp4_compressed_sparse_gb300 import build_lib, csa2
    build_lib.build()
    L = csa2.load()
    B, T, k, nblk = 3, 5000, 256, 64
    c, scores, q_pos = _scores(csa2, B, T, 16, seed=7)
    ref_idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    ref_pool = torch.empty((B, nblk), dtype=torch.int32, device="cuda")
    ref_cnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    csa2.topk(scores, 1, q_pos, k, ref_idx, csa2.topk_workspace(B, c.capacity, k, nblk),
              pool_out=ref_pool, pool_count=ref_cnt)
    for call in range(2):  # two calls in a row share the built-in scratch
        idx = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
        pool = torch.full((B, nblk), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        assert _call_noalloc(L, scores, q_pos, k, idx, pool, cnt) == 0
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx), f"call {call}: indices differ"
        assert torch.equal(pool, ref_pool) and torch.equal(cnt, ref_cnt), f"call {call}: pool differs"
    # a different problem right after (smaller k, pool-mode candidates)
    k2 = 32
    pool_in = ref_pool.clone()
    sc2 = torch.empty((B, nblk * 8), device="cuda")
    csa2.index_score(c, torch.randn((B, 16, 128), device="cuda").to(torch.bfloat16),
                     torch.rand((B, 16), device="cuda"), q_pos, sc2, pool=pool_in)
    ref2 = torch.empty((B, k2), dtype=torch.int32, device="cuda")
    csa2.topk(sc2, 1, q_pos, k2, ref2, csa2.topk_workspace(B, nblk * 8, k2), pool=pool_in)
    got2 = torch.empty((B, k2), dtype=torch.int32, device="cuda")
    assert _call_noalloc(L, sc2, q_pos, k2, got2, pool=pool_in) == 0
    torch.cuda.synchronize()
    assert torch.equal(got2, ref2)


def test_topk_noalloc_rejects_oversized_problem():
    from fp4_compressed_sparse_gb300 import build_lib, csa2
    build_lib.build()
    L = csa2.load()
    B, stride = 1024, 1 << 22
    # the same scratch csa2_topk would ask of its caller: far above the 4 MiB array
    assert L.csa2_topk_workspace_size(B, stride, 512, 0) > 4 * (4 << 20)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check rejects the call first
    st = L.csa2_topk_noalloc(fake, stride, B, 1, fake, None, 0, 8, 512, fake, 0, None, None, None, None)
    assert st == 7
    assert b"built-in" in L.csa2_last_error_detail()
