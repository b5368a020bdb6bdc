"""Helpers for the parity tests at the workloads' full sizes.

The CUDA side builds its caches through the C ABI in the same chunking as
bench.py.  The oracle encodes, from the same seeded rows, the indexer keys of
every visible position of a checked sequence (the score's only cache input)
and the latent records only where a check needs them (a "compact" oracle cache
whose slot j holds position positions[j]), so no oracle input comes from the
CUDA path.
"""
import numpy as np
import torch

from fp4_compressed_sparse_gb300 import csa2
from fp4_compressed_sparse_gb300 import workloads as wl

CHUNK = wl.CHUNK


def build_gpu_r1(W, extra_tokens=8):
    """Ratio-1 caches of W.batch sequences x W.context tokens, appended on the GPU."""
    cap = W.context + extra_tokens + 8
    c = csa2.Cache(W.batch, cap, ratio=1, swa_dtype=W.swa_dtype)
    rope = csa2.rope_table(W.theta, cap + 8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t0 in range(0, W.context, CHUNK):
        n = min(CHUNK, W.context - t0)
        kv = torch.stack([W.kv(b, t0, n, device="cuda") for b in range(W.batch)])
        ik = torch.stack([W.ik(b, t0, n, device="cuda") for b in range(W.batch)])
        csa2.kv_append(c, kv, ik, rope, err=err)
        del kv, ik
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return c, rope, err


def token_rows_at(W, stream, seq, positions, width):
    """Rows of the given token positions (any order), drawn chunk by chunk on the
    workload's device and copied to the host."""
    positions = np.asarray(positions, np.int64)
    out = np.zeros((positions.shape[0], width), np.float32)
    chunks = np.unique(positions // CHUNK)
    for ch in chunks:
        sel = np.nonzero(positions // CHUNK == ch)[0]
        blk = wl.normal((CHUNK, width), W.seed, stream, seq, int(ch), device=W.device)
        rows = torch.as_tensor(positions[sel] - ch * CHUNK, device=blk.device)
        out[sel] = blk[rows].cpu().numpy()
    return out


class Compact:
    """Oracle cache holding only the entries at `positions` (slot j = positions[j])."""

    def __init__(self, orc, W, seq, positions):
        self.positions = np.unique(np.asarray(positions, np.int64))
        self.slot = {int(p): j for j, p in enumerate(self.positions)}
        n = self.positions.shape[0]
        self.cache = orc.Cache(max(n, 1), swa_dtype=W.swa_dtype)
        kv = token_rows_at(W, wl.S_KV, seq, self.positions, 576)
        ik = token_rows_at(W, wl.S_IK, seq, self.positions, 128)
        c = self.cache
        for j, p in enumerate(self.positions):
            rec = orc.encode_entry(kv[j], ik[j], orc.rope_cs(W.theta, int(p)))
            for arr, val in zip((c.lat_codes, c.lat_scales, c.rope_codes, c.rope_scales,
                                 c.idx_codes, c.idx_scales), rec):
                arr[j] = val

    def remap(self, idx):
        return np.array([self.slot[int(i)] if i >= 0 else -1 for i in idx], np.int32)


def window_records(orc, W, seq, q_pos, n_tokens):
    """Oracle window rows of the query at q_pos: tokens max(0, q_pos-127) .. q_pos."""
    toks = orc.swa_tokens(q_pos, n_tokens)
    kv = token_rows_at(W, wl.S_KV, seq, toks, 576)
    recs = [orc.encode_swa(kv[j], orc.rope_cs(W.theta, t), W.swa_dtype) for j, t in enumerate(toks)]
    return np.array([r[0] for r in recs]), np.array([r[1] for r in recs])


def gpu_entries(c, seq, positions):
    """The GPU cache's record bytes of one sequence at the given positions."""
    pos = torch.as_tensor(np.asarray(positions, np.int64), device="cuda")
    ic, isc = c.idx_entries()
    return {
        "lat_codes": c.lat_codes[seq][pos].cpu().numpy(),
        "lat_scales": c.lat_scales[seq][pos].cpu().numpy(),
        "rope_codes": c.rope_codes[seq][pos].cpu().numpy(),
        "rope_scales": c.rope_scales[seq][pos].cpu().numpy(),
        "idx_codes": ic[seq][pos].cpu().numpy(),
        "idx_scales": isc[seq][pos].cpu().numpy(),
    }


def assert_entries_equal(c, seq, comp):
    g = gpu_entries(c, seq, comp.positions)
    for name, arr in g.items():
        ref = getattr(comp.cache, name)[:comp.positions.shape[0]]
        bad = np.argwhere(arr != ref)
        assert bad.size == 0, f"seq {seq} {name}: {len(bad)} bytes differ at entries " \
                              f"{comp.positions[bad[:3, 0]].tolist()}"


def oracle_keys(orc, W, seq, T):
    """The oracle's indexer-key records of positions 0..T-1 of one sequence,
    encoded from the workload's seeded key rows chunk by chunk."""
    kc = orc.KeyCache(T)
    for t0 in range(0, T, CHUNK):
        n = min(CHUNK, T - t0)
        orc.encode_keys(kc, t0, W.ik(seq, t0, n, device=W.device).cpu().numpy())
    return kc
