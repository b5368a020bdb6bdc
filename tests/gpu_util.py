"""Helpers shared by the GPU parity tests: build the CUDA cache and the oracle
cache from the same seeded inputs, and compare results."""
import numpy as np
import torch

from fp4_compressed_sparse_gb300 import csa2
from fp4_compressed_sparse_gb300 import workloads as wl

ATTN_TOL = 2e-3  # normwise relative error per (row, head), and |lse - lse_ref|


def u16(t):
    """bf16 torch tensor -> uint16 numpy (bit pattern)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def build_r1(orc, batch, n_tokens, swa_dtype, seed, chunks=None, in_bf16=False, cap=None,
             theta=10000.0, rope=None, kv_scale=1.0, entry_format=0):
    """Append n_tokens per sequence (in the given chunk sizes) on the GPU and in the
    oracle; the latent rows are multiplied by kv_scale (a power of two).
    Returns (gpu cache, [oracle caches], rope table, err word)."""
    cap = cap or n_tokens + 8
    c = csa2.Cache(batch, cap, ratio=1, swa_dtype=swa_dtype, entry_format=entry_format)
    rope = rope if rope is not None else csa2.rope_table(theta, cap + 8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    chunks = chunks or [n_tokens]
    oc = [orc.Cache(cap, swa_dtype=swa_dtype, entry_format=entry_format) for _ in range(batch)]
    t0 = 0
    for n in chunks:
        kv = torch.stack([wl.token_rows(seed, wl.S_KV, b, t0, n, 576) for b in range(batch)]) * kv_scale
        ik = torch.stack([wl.token_rows(seed, wl.S_IK, b, t0, n, 128) for b in range(batch)])
        if in_bf16:
            kv, ik = kv.to(torch.bfloat16), ik.to(torch.bfloat16)
        csa2.kv_append(c, kv.cuda(), ik.cuda(), rope, err=err)
        for b in range(batch):
            orc.append_r1(oc[b], kv[b].float().numpy(), ik[b].float().numpy(), theta)
        t0 += n
    torch.cuda.synchronize()
    return c, oc, rope, err


def cmp_rows(seed, seq, start, n):
    return [wl.token_rows(seed, s, seq, start, n, 704) for s in (wl.S_CA, wl.S_CB, wl.S_ZA, wl.S_ZB)]


def build_r2(orc, batch, n_tokens, swa_dtype, seed, chunks=None, cap=None, theta=10000.0,
             bias_scale=0.5, dbg=False, entry_format=0):
    """Ratio-2 appends on both sides.  Returns (gpu cache, oracle caches, rope, err,
    biases, gpu dbg rows per call, oracle dbg rows)."""
    cap = cap or n_tokens // 2 + 8
    c = csa2.Cache(batch, cap, ratio=2, swa_dtype=swa_dtype, entry_format=entry_format)
    rope = csa2.rope_table(theta, 2 * cap + 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = torch.Generator().manual_seed(seed + 991)
    ba = (torch.randn((2, 704), generator=g) * bias_scale).float()
    bb = (torch.randn((2, 704), generator=g) * bias_scale).float()
    chunks = chunks or [n_tokens]
    oc = [orc.Cache(cap, swa_dtype=swa_dtype, ratio=2, entry_format=entry_format) for _ in range(batch)]
    t0 = 0
    gdbg, odbg = [], [[] for _ in range(batch)]
    for n in chunks:
        rows = [torch.stack(x) for x in zip(*[cmp_rows(seed, b, t0, n) for b in range(batch)])]
        d = torch.zeros((batch, n // 2 + 1, 704), device="cuda") if dbg else None
        csa2.kv_append(c, rope_cs=rope, cmp=[r.cuda() for r in rows] + [ba.cuda(), bb.cuda()],
                       cmp_dbg=d, err=err)
        gdbg.append(d)
        for b in range(batch):
            orc.append_r2(oc[b], *[r[b].numpy() for r in rows], ba.numpy(), bb.numpy(), theta,
                          dbg=odbg[b])
        t0 += n
    torch.cuda.synchronize()
    return c, oc, rope, err, (ba, bb), gdbg, odbg


def assert_cache_equal(c, oc, n_entries, check_swa=True):
    ic, isc = c.idx_entries()
    planes = {"idx_codes": ic, "idx_scales": isc}
    for b, o in enumerate(oc):
        for name in ("lat_codes", "lat_scales", "rope_codes", "rope_scales", "idx_codes", "idx_scales"):
            if getattr(c, name, None) is None and name not in planes:
                continue  # a plane the entry format does not use
            g = planes.get(name, getattr(c, name, None))[b, :n_entries].cpu().numpy()
            ref = getattr(o, name)[:n_entries]
            bad = np.argwhere(g != ref)
            assert bad.size == 0, f"seq {b} {name}: {len(bad)} bytes differ, first {bad[:3].tolist()}"
        if check_swa:
            g = c.swa_codes[b].cpu().numpy()
            assert np.array_equal(g, o.swa_codes), f"seq {b} window codes differ"
            if c.swa_dtype == csa2.SWA_MXFP8:
                assert np.array_equal(c.swa_scales[b, :, :18].cpu().numpy(), o.swa_scales), \
                    f"seq {b} window scales differ"


def attn_close(out, lse, ref_out, ref_lse, tol=ATTN_TOL):
    """Normwise per-head check; returns the worst (out, lse) errors."""
    out = np.asarray(out, np.float64)
    ref_out = np.asarray(ref_out, np.float64)
    num = np.max(np.abs(out - ref_out), axis=-1)
    den = np.maximum(np.max(np.abs(ref_out), axis=-1), 1e-30)
    e_o = float(np.max(num / den))
    e_l = float(np.max(np.abs(np.asarray(lse, np.float64) - np.asarray(ref_lse, np.float64))))
    assert e_o <= tol, f"attention output normwise error {e_o:.3e} > {tol}"
    assert e_l <= tol, f"lse error {e_l:.3e} > {tol}"
    return e_o, e_l
