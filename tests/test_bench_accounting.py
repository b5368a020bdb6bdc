"""Host-side checks of the measurement arithmetic (no GPU): the algorithmic bytes
bench.py divides by its timings, rebuilt here from the per-unit record sizes, and
the attention workspace the C ABI asks for."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

# per-unit sizes: indexer key 64 B codes + 4 B scale; main entry 256 + 32 B plus the
# 32 + 4 B RoPE sidecar, read with its 4-byte index; MXFP8 window entry 576 + 18 B;
# bf16 query 576 dims; fp32 output 512 dims + lse
KEY, ENTRY, WIN8, WIN16 = 64 + 4, 256 + 32 + 32 + 4 + 4, 576 + 18, 576 * 2
Q, OUT = 576 * 2, 512 * 4


def test_decode_step_bytes_bench_workload():
    import bench
    B, T, H, H_I, k = 32, 65591, 64, 64, 512
    n = bench.decode_step_bytes(B, T, H, H_I, k, 1)
    assert n["keys"] == B * T * KEY == 142_726_016
    assert n["qidx"] == B * (H_I * 128 * 2 + H_I * 4)
    attn = B * (k * ENTRY + 128 * WIN8 + H * Q + H * OUT + H * 4)
    assert n["attn"] == attn
    # the figure the headline JSON line reports as algorithmic_bytes_per_step
    assert n["total"] == 157_748_928
    # a bf16 window doubles the window bytes only
    n16 = bench.decode_step_bytes(B, T, H, H_I, k, 0)
    assert n16["attn"] - n["attn"] == B * 128 * (WIN16 - WIN8)


def test_group_step_bytes_per_layer_role():
    import bench
    from fp4_compressed_sparse_gb300 import workloads as wl
    attn = 512 * ENTRY + 128 * WIN8 + 64 * Q + 64 * OUT
    qidx = 64 * 128 * 2 + 64 * 4
    W = wl.stack_1m(device="cpu")
    T = W.context + 3 + 4 // 2
    full = T * KEY + qidx + attn
    reindex = 2048 * 8 * KEY + 2048 * 4 + qidx + attn
    assert bench.group_step_bytes(W, T) == W.batch * (full + 4 * reindex + 3 * attn) == 635_728_544
    # the encoder group: ratio 2, so the Full layer scans half as many entries as tokens
    E = wl.encoder_decode(device="cpu")
    Te = (E.context + 3 + 6 // 2) // E.ratio
    assert bench.group_step_bytes(E, Te) == E.batch * (Te * KEY + qidx + 6 * attn) == 229_308_800


@pytest.fixture(scope="module")
def lib():
    from fp4_compressed_sparse_gb300 import build_lib, csa2
    build_lib.build()
    return csa2.load()


def test_attn_workspace_holds_every_segment_partial(lib):
    # a segment's partial: O [64][512] + (m, l) [64][2] fp32.  The segment count
    # is min(4, chunks) with chunks = ceil(k / 32) + 4 (the 128-token window) --
    # a function of k alone, so the workspace grows linearly with the batch
    part = 64 * (512 + 2) * 4
    assert lib.csa2_attn_workspace_size(1, 64, 512) == 4 * part + 256
    assert lib.csa2_attn_workspace_size(19, 64, 512) == 19 * 4 * part + 256
    assert lib.csa2_attn_workspace_size(32, 64, 512) == 32 * 4 * part + 256
    # 128 heads: two 64-head blocks per row; 48 heads: sized as one 64-head block
    assert lib.csa2_attn_workspace_size(1, 128, 512) == 2 * 4 * part + 256
    assert lib.csa2_attn_workspace_size(2, 48, 512) == 2 * 4 * part + 256
    # k = 1: one chunk of selected entries + 4 window chunks, still 4 segments
    assert lib.csa2_attn_workspace_size(1, 64, 1) == 4 * part + 256
