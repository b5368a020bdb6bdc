"""Seeded synthetic inputs for the CSA2 step.

This module only draws random numbers with the shapes and distributions of the
workloads (N(0,1) KV, queries and compression inputs, U(0,1) indexer head
weights, uniformly drawn candidate pools).  It holds none of the method's
arithmetic; both the CUDA path and the CPU oracle take their inputs from here.

Every draw is keyed by (seed, stream, sequence, chunk) so that any chunk can be
regenerated on its own, on the device it was first drawn on (torch's CPU and
CUDA generators give different streams, so a workload fixes its device).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

CHUNK = 8192  # tokens per independently seeded chunk

# stream ids
S_KV, S_IK, S_QIDX, S_W, S_Q, S_CA, S_CB, S_ZA, S_ZB, S_BA, S_BB, S_POOL, S_SINK = range(13)


def _seed(seed: int, *keys: int) -> int:
    s = (seed * 0x9E3779B1 + 0x632BE5AB) & ((1 << 63) - 1)
    for k in keys:
        s = (s * 1000003 + int(k) + 0x5851F42D) & ((1 << 63) - 1)
    return s


def _gen(device, seed, *keys):
    g = torch.Generator(device=device)
    g.manual_seed(_seed(seed, *keys))
    return g


def normal(shape, seed, *keys, device="cpu"):
    return torch.randn(shape, generator=_gen(device, seed, *keys), device=device,
                       dtype=torch.float32)


def uniform(shape, seed, *keys, device="cpu", lo=0.0, hi=1.0):
    u = torch.rand(shape, generator=_gen(device, seed, *keys), device=device, dtype=torch.float32)
    return u * (hi - lo) + lo


def token_rows(seed, stream, seq, start, n, width, device="cpu"):
    """N(0,1) rows [n, width] for tokens start..start+n-1 of one sequence."""
    out = torch.empty((n, width), dtype=torch.float32, device=device)
    t = start
    while t < start + n:
        c = t // CHUNK
        lo = c * CHUNK
        blk = normal((CHUNK, width), seed, stream, seq, c, device=device)
        a = t - lo
        b = min(CHUNK, start + n - lo)
        out[t - start:t - start + (b - a)] = blk[a:b]
        t = lo + b
    return out


@dataclass
class DecodeWorkload:
    """A decode-step workload: B sequences of `context` tokens each; the step
    appends token `context` and queries at that position."""
    name: str
    batch: int
    context: int
    heads: int
    index_heads: int
    topk: int
    swa_dtype: int  # 0 bf16, 1 MXFP8
    seed: int
    theta: float = 10000.0
    pool_blocks: int = 2048
    pool_block_size: int = 8
    layers: tuple = ("full",)  # sequence of "full" / "reindex" / "reuse"
    steps: int = 1
    ratio: int = 1  # 2: encoder-style cache, two tokens per entry (compression inputs below)
    device: str = "cpu"
    extra: dict = field(default_factory=dict)

    @property
    def sm_scale(self):
        return 1.0 / math.sqrt(576.0)

    # ----------------------------------------------------------- cache contents
    def kv(self, seq, start, n, device=None):
        return token_rows(self.seed, S_KV, seq, start, n, 576, device or self.device)

    def ik(self, seq, start, n, device=None):
        return token_rows(self.seed, S_IK, seq, start, n, 128, device or self.device)

    def cmp_rows(self, seq, start, n, device=None):
        """Ratio 2: (C^a, C^b, Z^a, Z^b) rows [n, 704] of one sequence's tokens start..start+n-1."""
        d = device or self.device
        return tuple(token_rows(self.seed, s, seq, start, n, 704, d) for s in (S_CA, S_CB, S_ZA, S_ZB))

    def bias(self, device=None):
        """Ratio 2: B^a, B^b [2, 704].  READING: zero positional bias (the workload states none)."""
        d = device or self.device
        return (torch.zeros((2, 704), device=d), torch.zeros((2, 704), device=d))

    # ----------------------------------------------------------- per step / layer
    def q_idx(self, step, layer, device=None):
        """bf16 [B, H_I, 128]"""
        return normal((self.batch, self.index_heads, 128), self.seed, S_QIDX, step, layer,
                      device=device or self.device).to(torch.bfloat16)

    def w(self, step, layer, device=None):
        """fp32 [B, H_I], U(0,1)"""
        return uniform((self.batch, self.index_heads), self.seed, S_W, step, layer,
                       device=device or self.device)

    def q(self, step, layer, device=None):
        """bf16 [B, H, 576] absorbed query (latent 512 + rotated RoPE 64)"""
        return normal((self.batch, self.heads, 576), self.seed, S_Q, step, layer,
                      device=device or self.device).to(torch.bfloat16)

    def pool(self, device="cpu"):
        """[B, pool_blocks] int32 ascending distinct block ids drawn uniformly from
        the blocks that cover the context (the Reindex workload's prior pool)."""
        nblk = self.context // self.pool_block_size
        out = torch.empty((self.batch, self.pool_blocks), dtype=torch.int32)
        for b in range(self.batch):
            g = _gen("cpu", self.seed, S_POOL, b)
            perm = torch.randperm(nblk, generator=g)[:self.pool_blocks]
            out[b] = torch.sort(perm).values.to(torch.int32)
        return out.to(device)


@dataclass
class PrefillWorkload:
    """Encoder-style chunked prefill: `prior` tokens already packed 2 per entry,
    then a chunk of `chunk` query tokens."""
    name: str
    prior: int
    chunk: int
    heads: int
    index_heads: int
    topk: int
    swa_dtype: int
    seed: int
    theta: float = 10000.0
    device: str = "cpu"

    @property
    def sm_scale(self):
        return 1.0 / math.sqrt(576.0)

    def cmp_rows(self, start, n, device=None):
        """(C^a, C^b, Z^a, Z^b) rows [n, 704] for tokens start..start+n-1."""
        d = device or self.device
        return tuple(token_rows(self.seed, s, 0, start, n, 704, d) for s in (S_CA, S_CB, S_ZA, S_ZB))

    def bias(self, device=None):
        """B^a, B^b [2, 704].  READING: zero positional bias (the workload states none)."""
        d = device or self.device
        return (torch.zeros((2, 704), device=d), torch.zeros((2, 704), device=d))

    def q_idx(self, device=None):
        return normal((self.chunk, self.index_heads, 128), self.seed, S_QIDX, 0,
                      device=device or self.device).to(torch.bfloat16)

    def w(self, device=None):
        return uniform((self.chunk, self.index_heads), self.seed, S_W, 0, device=device or self.device)

    def q(self, device=None):
        return normal((self.chunk, self.heads, 576), self.seed, S_Q, 0,
                      device=device or self.device).to(torch.bfloat16)


# The workloads: shapes, sizes and distributions of the decode / prefill
# configurations this library is measured on.
def tiny_decode(device="cpu"):
    return DecodeWorkload("tiny_decode_b1_t4096", batch=1, context=4096, heads=16, index_heads=4,
                          topk=64, swa_dtype=0, seed=0, device=device)


def full_decode(device="cuda"):
    return DecodeWorkload("full_decode_b32_t65536", batch=32, context=65536, heads=64,
                          index_heads=64, topk=512, swa_dtype=1, seed=1, device=device)


def full_decode_small(device="cuda"):
    """The Full-layer decode step at context 8,192: the attention and top-k launches
    have the shapes of full_decode, the cache is 8x smaller (small profiler captures)."""
    return DecodeWorkload("full_decode_b32_t8192", batch=32, context=8192, heads=64,
                          index_heads=64, topk=512, swa_dtype=1, seed=1, device=device)


def reindex_decode(device="cuda"):
    return DecodeWorkload("reindex_reuse3_b64_t262144", batch=64, context=262144, heads=64,
                          index_heads=64, topk=512, swa_dtype=1, seed=2,
                          layers=("reindex", "reuse", "reuse", "reuse"), device=device)


def reindex_masked_decode(device="cuda"):
    """reindex_decode with its Reindex layer in the published reference code's form:
    every visible position scored, the positions outside the pool masked, top-k of
    the whole row (same cache, pool and queries)."""
    return DecodeWorkload("reindex_masked_reuse3_b64_t262144", batch=64, context=262144, heads=64,
                          index_heads=64, topk=512, swa_dtype=1, seed=2,
                          layers=("reindex_masked", "reuse", "reuse", "reuse"), device=device)


def prefill_chunk(device="cuda"):
    return PrefillWorkload("prefill_q8192_prior131072_r2", prior=131072, chunk=8192, heads=64,
                           index_heads=64, topk=512, swa_dtype=1, seed=3, device=device)


def prefill_chunk_small(device="cuda"):
    """The chunked prefill with a chunk of 512 queries against the same 131,072 prior
    tokens: one block of queries per launch, for small profiler captures."""
    return PrefillWorkload("prefill_q512_prior131072_r2", prior=131072, chunk=512, heads=64,
                           index_heads=64, topk=512, swa_dtype=1, seed=3, device=device)


def encoder_decode(device="cuda"):
    """An encoder group at decode: ratio-2 caches of 131,072 tokens (65,536 entries),
    one token appended per step through the compression buffer, a Full layer and
    five Reuse layers."""
    return DecodeWorkload("encoder_full_reuse5_b32_t131072_r2", batch=32, context=131072, heads=64,
                          index_heads=64, topk=512, swa_dtype=1, seed=5, ratio=2,
                          layers=("full", "reuse", "reuse", "reuse", "reuse", "reuse"), device=device)


def stack_1m(device="cuda"):
    return DecodeWorkload("stack_b8_t1048576_100steps", batch=8, context=1048576, heads=64,
                          index_heads=64, topk=512, swa_dtype=1, seed=4, steps=100,
                          layers=("full", "reindex", "reindex", "reindex", "reindex", "reuse",
                                  "reuse", "reuse"), device=device)
