// csa2_attn.cu -- sparse absorbed-query attention over the selected FP4 entries
// plus the sliding window, with an optional attention sink.
//
// [P5] "DeepSeek-V4: Towards Highly Efficient Million-Token Context
// Intelligence" §2.3.1 "Shared Key-Value MQA" (each selected entry is key and
// value, shared by all heads), §2.3.3 (window branch; sink exp(z'_h) in the
// denominator); [P2] "DeepSeek Multi-Head Latent Attention(MLA) 해부" §4
// (absorbed query: the logit is q_lat . c + q_rope . k_rope, the value is the
// 512-dim latent c).
//
// Two kernels with the same entry gather, dequantisation and segment schedule:
// k_attn (below) for decode rows, with both contractions on mma.sync and O in
// registers; k_attn_tc (further below) for one-segment rows (the chunked
// prefill, a query's whole entry list in one CTA), with both contractions on
// the tcgen05 tensor cores and O in tensor memory.
//
// k_attn: one CTA = (some segments of a row's entry list, up to 64 heads).
// Every head shares the entries, so each entry is dequantised once per CTA:
//   producer warps (4)  gather 32 entries at a time and dequantise them into a
//                       two-stage fp16 ring: E2M1 pairs by cvt.f16x2.e2m1x2, times
//                       the E4M3 scale (exact: at most 6 significant bits, >= 2^-10);
//                       V4-format entries (E4M3 latent with E8M0 scales, bf16
//                       RoPE dims) like the 8-bit / bf16 window entries;
//                       window MXFP8 / bf16 entries, scaled by a power of two
//                       2^-sigma_j only if they would not fit fp16
//   consumer warps      S = Q K^T (mma.sync m16n8k16 f16, fp32 accumulate; a
//   (heads / 8)         warp takes 16 heads x the chunk's 32 entries over one half
//                       of the 576 dims, the two halves summed by the softmax),
//                       online softmax in the log2 domain, O += P V with the fp32
//                       O tile in registers
// The query is held as fp16 with a power-of-two scale per head (exact for bf16
// values within 2^24 of the head's maximum).  Stage handover uses mbarriers
// with bounded waits (CSA2_DEVERR_TIMEOUT if one runs out).
//
// Batch-invariant schedule ([P5] §3.3: a token's output must not depend on the
// batch it was computed in, so the accumulation order may not follow the
// launch shape).  A row's entry list is cut into S segments, S fixed by k and
// the window alone (chunk c of 32 entries belongs to segment c % S).  Each
// segment gets its own online softmax and leaves an unnormalised partial
// (O, m, l); the row's output merges the S partials in segment order
// (flash-decoding LSE merge, then the sink).  Only the number G of CTAs a row
// is spread over follows the batch (enough CTAs to fill the SMs): CTA g of the
// row computes segments g, g + G, ... one after the other, writes their partials
// to a workspace that stays in L2, and after a cluster barrier (the row's G CTAs
// are one thread-block cluster) merges a slice of the heads -- the same
// arithmetic in the same order for any G, so the bits do not change with it.
#include <cuda_fp16.h>

#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {
namespace {

constexpr int kE = 32;            // entries per chunk
constexpr int kQS = kDqk + 8;     // fp16 row stride of Q and of the entry tiles (1168 B: conflict-free ldmatrix)
constexpr int kPS = kE + 8;       // fp16 row stride of P (80 B)
constexpr int kSS = kE + 8;       // fp32 row stride of the partial logits (conflict-free float2 stores)
constexpr int kProdThreads = 128; // four producer warps
constexpr int kHeadBlock = 64;    // heads per CTA at most (16 or 32 when small batches need more CTAs)
constexpr uint32_t kWaitIters = 200;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxChunks = (CSA2_MAX_TOPK + kWin) / kE;  // chunks of the longest entry list (68)

template <int HP>
struct __align__(16) AttnSmem {
  __half q[HP][kQS];
  __half kv[2][kE][kQS];
  float s[2][HP][kSS]; // partial logits over dims 0..287 and 288..575
  __half p[HP][kPS];
  float qf[HP];        // logit factor of head h: 2^e_h * sm_scale * log2(e)
  float alpha[HP];     // this chunk's rescale of O
  float fin[HP][2];    // m, l per head after the last chunk
  float sig[2][kE];    // 2^sigma_j of entry j of a stage; 0 = empty entry
  int16_t chunk_id[kMaxChunks];  // the CTA's chunks in processing order
  int8_t seg_end[kMaxChunks];    // the segment a chunk ends, or -1
  int nchunks;
  __align__(8) uint64_t full[2];
  __align__(8) uint64_t empty[2];
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t x, uint32_t y) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&x), *reinterpret_cast<__half2 *>(&y));
  return *reinterpret_cast<uint32_t *>(&r);
}
// two E4M3 codes (low byte -> low half) to fp16, exactly
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two_bytes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(static_cast<uint16_t>(two_bytes)));
  return r;
}
// two E2M1 codes (the low byte of `byte`; low nibble -> low half) to fp16, exactly
__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n" : "=r"(r) : "r"(byte));
  return r;
}
__device__ __forceinline__ uint32_t h2_splat(float v) {
  __half2 h = __float2half2_rn(v);
  return *reinterpret_cast<uint32_t *>(&h);
}
constexpr int kMaxSeg = 8;  // segments of a row at most; also the most CTAs per row (one portable cluster)
constexpr int kSegments = 4;  // segments of a decode row (fewer when its entry list has fewer chunks)

// every non-exited thread of the cluster
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// a float2 / float4 written by another CTA of the cluster before a cluster barrier (L2, not L1)
__device__ __forceinline__ float4 ld_cg4(const float *p) { return __ldcg(reinterpret_cast<const float4 *>(p)); }
__device__ __forceinline__ float2 ld_cg2(const float *p) { return __ldcg(reinterpret_cast<const float2 *>(p)); }

__device__ __forceinline__ void bar_consumers(int n) { asm volatile("bar.sync 1, %0;\n" ::"r"(n) : "memory"); }
// consumer barrier returning the AND of v over the consumer threads
__device__ __forceinline__ int bar_consumers_and(int n, int v) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.s32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v), "r"(n)
      : "memory");
  return r;
}

// Warp-uniform bounded wait on an mbarrier phase.
__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity, int32_t *err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) {
    ok = tc::mbar_wait_bounded(bar, parity, kWaitIters) ? 1 : 0;
    if (!ok) raise_err(err, CSA2_DEVERR_TIMEOUT);
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// The row's entry list: the k selected cache entries padded with empties to
// kpad = ceil(k / 32) * 32, then the 128 window tokens; chunk c = entries
// 32c .. 32c + 31.  Segment s of S holds chunks s, s + S, s + 2S, ... so every
// segment gets its share of the window.
// Kind of entry j: 0 empty, 1 cache entry, 2 window ring slot, 3 window row
// of the call.  `sel` is the raw index of a selected entry (read ahead).
__device__ __forceinline__ int entry_kind(const AttnArgs &a, int seq, int j, int kpad, int32_t sel, int64_t qpos,
                                          int64_t T, int64_t ntok, int64_t lin_base, int64_t &src) {
  src = 0;
  if (j < kpad) {
    if (j >= a.k || sel < 0) return 0;
    if (sel >= T || sel >= a.cap) {
      raise_err(a.err, CSA2_DEVERR_INDEX);
      return 0;
    }
    src = phys_entry(a.map, seq, sel);
    if (src < 0) {  // a page id outside the pool
      raise_err(a.err, CSA2_DEVERR_INDEX);
      return 0;
    }
    return 1;
  }
  const int64_t tok = qpos - (kWin - 1) + (j - kpad);
  if (tok < 0 || tok >= ntok || tok > qpos) return 0;
  if (tok >= lin_base) {
    src = tok - lin_base;
    return 3;
  }
  src = static_cast<int64_t>(a.ring_single ? 0 : seq) * kWin + (tok % kWin);
  return 2;
}

// Raw bytes of one FP4 cache entry held by one producer thread (its quarter).
struct Fp4Raw {
  uint2 cw[9];   // code bytes of units q4 + 4i (i < 8) and RoPE unit q4
  uint4 s0, s1;  // the 32 latent scale bytes
  uint32_t rsc;  // RoPE scale byte of group q4
};

__device__ __forceinline__ void load_fp4(const AttnArgs &a, int64_t src, int q4, Fp4Raw &r) {
  const uint2 *lc = reinterpret_cast<const uint2 *>(a.lat_codes + src * 256);
#pragma unroll
  for (int i = 0; i < 8; ++i) r.cw[i] = lc[q4 + 4 * i];
  r.cw[8] = reinterpret_cast<const uint2 *>(a.rope_codes + src * 32)[q4];
  const uint4 *ls = reinterpret_cast<const uint4 *>(a.lat_scales + src * 32);
  r.s0 = ls[0];
  r.s1 = ls[1];
  r.rsc = a.rope_scales[src * 4 + q4];
}

// Dequantises this producer thread's quarter of one entry of kind `kind` (at
// src) into fp16 through put(u, lo, hi): 16-dim unit u (dims 16u .. 16u + 7 in
// lo, the next 8 in hi), units q4, q4 + 4, ... of the 36.  FP4 entries are exact
// (E2M1 pairs by cvt.f16x2.e2m1x2, times the E4M3 scale); V4 entries and window
// entries are scaled by a power of two 2^-sigma only when they would not fit
// fp16.  Returns 2^sigma, 0 for an empty entry.  The four threads of an entry
// (qmask) take the same branch.
template <class Put>
__device__ __forceinline__ float dequant_entry(const AttnArgs &a, int kind, int64_t src, const Fp4Raw &raw, int q4,
                                               uint32_t qmask, bool fp8, Put put) {
  float sig = 0.0f;
  if (kind == 1 && fp8) {
    // V4 entry: 512 E4M3 codes with an E8M0 per 32, then 64 bf16 RoPE dims;
    // scaled by a power of two 2^-sigma only if they would not fit fp16
    const uint8_t *lc = a.lat_codes + src * 512;
    const uint4 sv = *reinterpret_cast<const uint4 *>(a.lat_scales + src * 16);
    const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
    uint32_t mx = 0;
#pragma unroll
    for (int g = 0; g < 16; ++g) mx = max(mx, (sw[g >> 2] >> (8 * (g & 3))) & 0xFFu);
    const uint4 *rc = reinterpret_cast<const uint4 *>(a.rope_codes + src * 128 + 32 * q4);
    const uint4 r0 = rc[0], r1 = rc[1];
    const uint32_t rw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    float ramax = 0.0f;
#pragma unroll
    for (int b = 0; b < 8; ++b)
      ramax = fmaxf(ramax, fmaxf(fabsf(__uint_as_float(rw[b] << 16)), fabsf(__uint_as_float(rw[b] & 0xFFFF0000u))));
    ramax = fmaxf(ramax, __shfl_xor_sync(qmask, ramax, 1));
    ramax = fmaxf(ramax, __shfl_xor_sync(qmask, ramax, 2));
    // latent values < 448 * 2^(mx-127), RoPE values <= ramax: both below 2^16 after 2^-sigma
    const int s_lat = static_cast<int>(mx) - 134;
    const int s_rope = ramax > 0.0f ? floor_log2f(ramax) - 14 : 0;
    const int sigma = min(15, max(0, max(s_lat, s_rope)));
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      const int u = q4 + 4 * i;  // 16 latent dims, half of scale block u / 2
      const uint4 cw = reinterpret_cast<const uint4 *>(lc)[u];
      const int wi = u >> 3;  // scale word of unit u (a select chain: no local array)
      const uint32_t swu = wi == 0 ? sv.x : wi == 1 ? sv.y : wi == 2 ? sv.z : sv.w;
      const int sc = static_cast<int>((swu >> (8 * ((u >> 1) & 3))) & 0xFFu);
      const int kx = sc - 127 - sigma;
      const uint32_t m2 = h2_splat(kx < -24 ? 0.0f : pow2f(kx));
      const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
      uint32_t o[8];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        o[2 * b] = hmul2u(e4m3x2_to_h2(w[b] & 0xFFFFu), m2);
        o[2 * b + 1] = hmul2u(e4m3x2_to_h2(w[b] >> 16), m2);
      }
      put(u, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
    }
    {  // RoPE unit 32 + q4: 16 bf16 dims
      const float inv = pow2f(-sigma);
      uint32_t o[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        __half2 t2 = __floats2half2_rn(__fmul_rn(__uint_as_float(rw[b] << 16), inv),
                                       __fmul_rn(__uint_as_float(rw[b] & 0xFFFF0000u), inv));
        o[b] = *reinterpret_cast<uint32_t *>(&t2);
      }
      put(32 + q4, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
    }
    sig = pow2f(sigma);
  } else if (kind == 1) {
    // FP4 entry: unit u < 32 = latent dims 16u.. (8 code bytes, scale u), u = 32 + q4 the RoPE group q4
    const uint32_t sw[8] = {raw.s0.x, raw.s0.y, raw.s0.z, raw.s0.w, raw.s1.x, raw.s1.y, raw.s1.z, raw.s1.w};
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const int u = i < 8 ? q4 + 4 * i : 32 + q4;
      // unit q4 + 4 i has scale byte q4 of word i (a static index: no local array)
      const uint32_t sb = i < 8 ? (sw[i] >> (8 * q4)) & 0xFFu : raw.rsc;
      const uint32_t s2 = e4m3x2_to_h2(sb | (sb << 8));
      uint32_t o[8];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        o[b] = hmul2u(e2m1x2_to_h2(raw.cw[i].x >> (8 * b)), s2);
        o[4 + b] = hmul2u(e2m1x2_to_h2(raw.cw[i].y >> (8 * b)), s2);
      }
      put(u, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
    }
    sig = 1.0f;
  } else if (kind == 2 || kind == 3) {
    const bool ring = kind == 2;
    const int rec = a.swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152;
    const uint8_t *cb = (ring ? a.ring_codes : a.lin_codes) + src * rec;
    if (a.swa_dtype == CSA2_SWA_MXFP8) {
      const uint4 *sp = reinterpret_cast<const uint4 *>((ring ? a.ring_scales : a.lin_scales) +
                                                        src * kSwaScaleStride);
      const uint4 s0 = sp[0], s1 = sp[1];
      const uint32_t sw[5] = {s0.x, s0.y, s0.z, s0.w, s1.x};
      uint32_t mx = 0;
#pragma unroll
      for (int g = 0; g < 18; ++g) mx = max(mx, (sw[g >> 2] >> (8 * (g & 3))) & 0xFFu);
      // values < 448 * 2^(sc-127): keep them below 2^16 with sigma >= 0
      const int sigma = min(15, max(0, static_cast<int>(mx) - 134));
#pragma unroll 1
      for (int i = 0; i < 9; ++i) {
        const int u = q4 + 4 * i;
        const uint4 cw = reinterpret_cast<const uint4 *>(cb)[u];
        const int wi = u >> 3;  // scale word of unit u (a select chain: no local array)
        const uint32_t swu = wi == 0 ? sw[0] : wi == 1 ? sw[1] : wi == 2 ? sw[2] : wi == 3 ? sw[3] : sw[4];
        const int sc = static_cast<int>((swu >> (8 * ((u >> 1) & 3))) & 0xFFu);
        const int kx = sc - 127 - sigma;
        const uint32_t m2 = h2_splat(kx < -24 ? 0.0f : pow2f(kx));
        const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
        uint32_t o[8];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          o[2 * b] = hmul2u(e4m3x2_to_h2(w[b] & 0xFFFFu), m2);
          o[2 * b + 1] = hmul2u(e4m3x2_to_h2(w[b] >> 16), m2);
        }
        put(u, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
      }
      sig = pow2f(sigma);
    } else {
      const uint4 *cw = reinterpret_cast<const uint4 *>(cb);
      float amax = 0.0f;
#pragma unroll 1
      for (int i = 0; i < 9; ++i) {
        const int u = q4 + 4 * i;
        const uint4 v0 = cw[2 * u], v1 = cw[2 * u + 1];
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int b = 0; b < 8; ++b)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[b] << 16)), fabsf(__uint_as_float(w[b] & 0xFFFF0000u))));
      }
      amax = fmaxf(amax, __shfl_xor_sync(qmask, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(qmask, amax, 2));
      const int sigma = amax > 0.0f ? min(15, max(0, floor_log2f(amax) - 14)) : 0;
      const float inv = pow2f(-sigma);
#pragma unroll 1
      for (int i = 0; i < 9; ++i) {
        const int u = q4 + 4 * i;
        const uint4 v0 = cw[2 * u], v1 = cw[2 * u + 1];
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t o[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          __half2 t2 = __floats2half2_rn(__fmul_rn(__uint_as_float(w[b] << 16), inv),
                                         __fmul_rn(__uint_as_float(w[b] & 0xFFFF0000u), inv));
          o[b] = *reinterpret_cast<uint32_t *>(&t2);
        }
        put(u, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
      }
      sig = pow2f(sigma);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const int u = q4 + 4 * i;
      put(u, make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0));
    }
  }
  return sig;
}

// L2 prefetch of this producer thread's share of one entry's record (kind, src
// as from entry_kind): the lines its dequantisation will read.
__device__ __forceinline__ void l2_line(const void *p) { asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p)); }
__device__ __forceinline__ void prefetch_entry(const AttnArgs &a, int kind, int64_t src, int q4, bool fp8) {
  if (kind == 1) {
    if (fp8) {
      l2_line(a.lat_codes + src * 512 + 128 * q4);
      if (q4 == 0) l2_line(a.lat_scales + src * 16);
      if (q4 == 1) l2_line(a.rope_codes + src * 128);
    } else {
      if (q4 < 2) l2_line(a.lat_codes + src * 256 + 128 * q4);
      if (q4 == 2) l2_line(a.lat_scales + src * 32);
      if (q4 == 3) {
        l2_line(a.rope_codes + src * 32);
        l2_line(a.rope_scales + src * 4);
      }
    }
  } else if (kind == 2 || kind == 3) {
    const bool ring = kind == 2;
    const int rec = a.swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152;
    const uint8_t *cb = (ring ? a.ring_codes : a.lin_codes) + src * rec;
    for (int off = 128 * q4; off < rec; off += 512) l2_line(cb + off);
    if (q4 == 3) l2_line(cb + rec - 1);
    if (q4 == 0 && a.swa_dtype == CSA2_SWA_MXFP8) l2_line((ring ? a.ring_scales : a.lin_scales) + src * kSwaScaleStride);
  }
}

// load_fp4 with every load issued where it stands (volatile): the compiler may
// not sink a prefetch for a later chunk down to its first use
__device__ __forceinline__ uint2 ldv2(const void *p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ldv4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldv1(const void *p) {
  uint32_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];\n" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void load_fp4_early(const AttnArgs &a, int64_t src, int q4, Fp4Raw &r) {
  const uint8_t *lc = a.lat_codes + src * 256;
#pragma unroll
  for (int i = 0; i < 8; ++i) r.cw[i] = ldv2(lc + 8 * (q4 + 4 * i));
  r.cw[8] = ldv2(a.rope_codes + src * 32 + 8 * q4);
  r.s0 = ldv4(a.lat_scales + src * 32);
  r.s1 = ldv4(a.lat_scales + src * 32 + 16);
  r.rsc = ldv1(a.rope_scales + src * 4 + q4);
}

// Partial results of one (row, head block, segment) in the workspace: O
// [HP][512] then (m, l) [HP][2], fp32.
template <int HP>
__host__ __device__ constexpr size_t part_floats() { return static_cast<size_t>(HP) * (kLat + 2); }

// The merge of a row's segments, run by every consumer warp of every CTA of
// the row after the cluster barrier: CTA `cta` of G merges heads cta, cta + G,
// ... from the partials of all n_seg segments (n_seg <= kS), always in segment
// order.  A warp takes kH of its heads at a time and requests every partial
// value of them -- the O rows and the (m, l) pairs -- before it uses any.
// Flash-decoding LSE merge, then the sink.
template <int kS, int kH, int HP>
__device__ __forceinline__ void merge_heads(const AttnArgs &a, const float *part, int row, int hbase, int nh,
                                            int cta, int n_cta, int n_seg, int warp, int nwarps, int lane) {
  const int stride = n_cta * nwarps;
  for (int hl0 = cta + n_cta * warp; hl0 < nh; hl0 += stride * kH) {
    float4 v[kH][kS][kLat / 128];
    float ms[kH], ls[kH];
#pragma unroll
    for (int j = 0; j < kH; ++j) {
      const int hl = hl0 + stride * j;  // warp-uniform
#pragma unroll
      for (int sp = 0; sp < kS; ++sp)
#pragma unroll
        for (int c = 0; c < kLat / 128; ++c)
          v[j][sp][c] = hl < nh && sp < n_seg
                            ? ld_cg4(part + sp * part_floats<HP>() + static_cast<size_t>(hl) * kLat + 128 * c + 4 * lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      ms[j] = -INFINITY;
      ls[j] = 0.0f;
      if (hl < nh && lane < n_seg) {  // lane s < n_seg holds segment s's (m, l)
        const float2 ml = ld_cg2(part + lane * part_floats<HP>() + static_cast<size_t>(HP) * kLat + 2 * hl);
        ms[j] = ml.x;
        ls[j] = ml.y;
      }
    }
#pragma unroll
    for (int j = 0; j < kH; ++j) {
      const int hl = hl0 + stride * j;
      if (hl >= nh) break;
      const int h = hbase + hl;
      float M = ms[j];
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
      const float s2 = a.sink ? a.sink[h] * kLog2e : -INFINITY;
      M = fmaxf(M, s2);
      const float f = (M == -INFINITY || ms[j] == -INFINITY) ? 0.0f : exp2f(ms[j] - M);
      float L = ls[j] * f;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
      if (a.sink && M != -INFINITY) L += exp2f(s2 - M);
      const float inv = L > 0.0f ? 1.0f / L : 0.0f;
      float fs[kS];
#pragma unroll
      for (int sp = 0; sp < kS; ++sp) fs[sp] = __shfl_sync(0xffffffffu, f, sp) * inv;
      float *out = a.out + (static_cast<size_t>(row) * a.heads + h) * kLat;
#pragma unroll
      for (int c = 0; c < kLat / 128; ++c) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int sp = 0; sp < kS; ++sp) {
          acc.x += v[j][sp][c].x * fs[sp];
          acc.y += v[j][sp][c].y * fs[sp];
          acc.z += v[j][sp][c].z * fs[sp];
          acc.w += v[j][sp][c].w * fs[sp];
        }
        *reinterpret_cast<float4 *>(out + 128 * c + 4 * lane) = acc;
      }
      if (lane == 0) a.lse[static_cast<size_t>(row) * a.heads + h] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
  }
}

template <int HP>
__global__ void __launch_bounds__(HP * 4 + kProdThreads, 1) k_attn(AttnArgs a, int n_cta, int n_seg, float *part_ws) {
  constexpr int kCons = HP * 4;         // consumer threads: HP / 8 warps
  constexpr int kDW = 4096 / HP;        // output dims per consumer warp
  constexpr int kNT = kDW / 8;          // n8 tiles per consumer warp
  constexpr int kMT = HP / 16;          // m16 tiles (head groups)
  extern __shared__ __align__(128) uint8_t smem_raw[];
  AttnSmem<HP> &sm = *reinterpret_cast<AttnSmem<HP> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, row = blockIdx.y, hbase = blockIdx.z * HP;
  const int nh = min(HP, a.heads - hbase);
  const int seq = a.cache_seq < 0 ? row : a.cache_seq;
  const int kpad = (a.k + kE - 1) / kE * kE;
  const int total_chunks = (kpad + kWin) / kE;

  // ---- set-up: barriers, and this CTA's chunks: segments cta, cta + G, ...,
  // each segment's chunks in ascending order
  if (tid == 0) {
    tc::mbar_init(&sm.full[0], kProdThreads);
    tc::mbar_init(&sm.full[1], kProdThreads);
    tc::mbar_init(&sm.empty[0], kCons);
    tc::mbar_init(&sm.empty[1], kCons);
    tc::fence_mbar_init();
    int n = 0;
    for (int sg = cta; sg < n_seg; sg += n_cta) {
      for (int ch = sg; ch < total_chunks && n < kMaxChunks; ch += n_seg) {
        sm.chunk_id[n] = static_cast<int16_t>(ch);
        sm.seg_end[n] = -1;
        ++n;
      }
      if (n > 0) sm.seg_end[n - 1] = static_cast<int8_t>(sg);
    }
    sm.nchunks = n;
  }
  // launched as a programmatic dependent of the previous kernel: the block is
  // resident and set up while that grid drains, and nothing in memory (query,
  // positions, token counts, selection) is read before it is complete
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  __syncthreads();  // barriers and the chunk list ready
  const int nchunks = sm.nchunks;
  const int64_t qpos = a.q_pos[row];
  const int64_t T = qpos / a.ratio;
  const int64_t ntok = a.n_tokens[seq];
  const int64_t lin_base = a.lin_base ? *a.lin_base : INT64_MAX;

  if (tid >= kCons) {
    // ================================================================ producers
    const int pt = tid - kCons;
    const int e = pt >> 2, q4 = pt & 3;
    const uint32_t qmask = 0xFu << (lane & ~3);  // the four lanes of this entry
    const int32_t *idx_row = a.idx + static_cast<size_t>(row) * a.k;
    // software pipeline: once chunk c is handed over, the raw bytes of chunk
    // c+1 and the indices of chunk c+2 are requested; they land while this
    // producer waits for a free stage
    auto sel_of = [&](int i) -> int32_t {  // selected index of entry e of local chunk i, or -1
      const int j = sm.chunk_id[i] * kE + e;
      return j < a.k ? idx_row[j] : -1;
    };
    int64_t src = 0;
    int kind = 0;
    Fp4Raw raw;
    int32_t sel_next = -1;
    const bool fp8 = a.entry_format == CSA2_ENTRY_FP8;
    if (nchunks > 0) {
      kind = entry_kind(a, seq, sm.chunk_id[0] * kE + e, kpad, sel_of(0), qpos, T, ntok, lin_base, src);
      if (kind == 1 && !fp8) load_fp4(a, src, q4, raw);
      if (nchunks > 1) sel_next = sel_of(1);
    }
    bool dead = false;
    for (int c = 0; c < nchunks; ++c) {
      const int st = c & 1;
      if (c >= 2 && !dead) dead = !wait_warp(&sm.empty[st], ((c - 2) >> 1) & 1, a.err);
      if (!dead) {
        uint4 *dst = reinterpret_cast<uint4 *>(&sm.kv[st][e][0]);  // 16-dim unit u at dst[2u], dst[2u+1]
        const float sig = dequant_entry(a, kind, src, raw, q4, qmask, fp8, [&](int u, uint4 lo, uint4 hi) {
          dst[2 * u] = lo;
          dst[2 * u + 1] = hi;
        });
        if (q4 == 0) sm.sig[st][e] = sig;
      }
      tc::mbar_arrive(&sm.full[st]);
      if (c + 1 < nchunks) {
        kind = entry_kind(a, seq, sm.chunk_id[c + 1] * kE + e, kpad, sel_next, qpos, T, ntok, lin_base, src);
        if (kind == 1 && !fp8) load_fp4(a, src, q4, raw);
        if (c + 2 < nchunks) sel_next = sel_of(c + 2);
      }
    }
    if (n_seg > 1) cluster_sync();  // the consumers' cluster barrier, matched here
    return;
  }

  // ================================================================== consumers
  // the query to fp16 in sm.q with a power-of-two scale per head: |q * 2^-e| <
  // 2^15, exact for every bf16 value >= amax * 2^-24.  Warp w converts heads
  // w, w + HP/8, ... (eight of them), lane l the bf16 pairs l, l + 32, ... of a
  // head; every raw value of the warp's heads is requested from global memory
  // before any is used (one round trip), and the eight heads' reductions run
  // interleaved.
  {
    constexpr int kQW = 8;              // heads per consumer warp
    constexpr int kQP = kDqk / 2 / 32;  // bf16 pairs per lane per head (9)
    static_assert(kQW * (kCons / 32) == HP, "every head has one converting warp");
    uint32_t raw[kQW][kQP];
#pragma unroll
    for (int j = 0; j < kQW; ++j) {
      const int h = warp + (kCons / 32) * j;
      const uint32_t *gq =
          reinterpret_cast<const uint32_t *>(a.q + (static_cast<size_t>(row) * a.heads + hbase + h) * kDqk);
#pragma unroll
      for (int i = 0; i < kQP; ++i) raw[j][i] = h < nh ? __ldg(gq + lane + 32 * i) : 0u;
    }
    float amax[kQW];
#pragma unroll
    for (int j = 0; j < kQW; ++j) {
      amax[j] = 0.0f;
#pragma unroll
      for (int i = 0; i < kQP; ++i)
        amax[j] = fmaxf(amax[j], fmaxf(fabsf(__uint_as_float(raw[j][i] << 16)),
                                       fabsf(__uint_as_float(raw[j][i] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1)
#pragma unroll
      for (int j = 0; j < kQW; ++j) amax[j] = fmaxf(amax[j], __shfl_xor_sync(0xffffffffu, amax[j], o));
#pragma unroll
    for (int j = 0; j < kQW; ++j) {
      const int h = warp + (kCons / 32) * j;
      int ex = amax[j] > 0.0f ? floor_log2f(amax[j]) - 14 : 0;
      ex = max(ex, -110);
      const float inv = pow2f(-ex);
      uint32_t *dq = reinterpret_cast<uint32_t *>(&sm.q[h][0]);
#pragma unroll
      for (int i = 0; i < kQP; ++i) {
        __half2 t2 = __floats2half2_rn(__fmul_rn(__uint_as_float(raw[j][i] << 16), inv),
                                       __fmul_rn(__uint_as_float(raw[j][i] & 0xFFFF0000u), inv));
        dq[lane + 32 * i] = *reinterpret_cast<uint32_t *>(&t2);
      }
      if (lane == 0) sm.qf[h] = h < nh ? pow2f(ex) * a.sm_scale * kLog2e : 0.0f;
    }
  }
  bar_consumers(kCons);

  const int g = lane >> 2, t = lane & 3;
  float o[kMT][kNT][4];
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.0f;
  const int sh = tid >> 2, sq = tid & 3;  // softmax: head sh, entries 8 sq .. 8 sq + 7
  float m_run = -INFINITY, l_run = 0.0f;
  bool dead = false;
  const int hg = warp >> 1, kh = warp & 1;  // QK: heads 16 hg.., dims 288 kh..
  const int d0 = warp * kDW;                // PV: dims d0 .. d0 + kDW - 1

  for (int c = 0; c < nchunks; ++c) {
    const int st = c & 1;
    if (!dead) dead = !wait_warp(&sm.full[st], (c >> 1) & 1, a.err);
    if (!dead) {
      // ---- partial logits of heads 16hg.. x the 32 entries over dims 288kh..
      // (four independent accumulator chains, one per n8 tile of entries)
      float acc[4][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t qa = smem_u32(&sm.q[16 * hg + (lane & 15)][kh * (kDqk / 2) + (lane >> 4) * 8]);
      const uint32_t kb = smem_u32(&sm.kv[st][(lane & 7) + ((lane >> 4) << 3)][kh * (kDqk / 2) + ((lane >> 3) & 1) * 8]);
#pragma unroll 3
      for (int kk = 0; kk < kDqk / 32; ++kk) {
        uint32_t af[4], b0, b1, b2, b3, c0, c1, c2, c3;
        ldsm_x4(qa + kk * 32, af[0], af[1], af[2], af[3]);
        ldsm_x4(kb + kk * 32, b0, b1, b2, b3);
        ldsm_x4(kb + 16 * kQS * 2 + kk * 32, c0, c1, c2, c3);
        mma_f16(acc[0], af, b0, b1);
        mma_f16(acc[1], af, b2, b3);
        mma_f16(acc[2], af, c0, c1);
        mma_f16(acc[3], af, c2, c3);
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          *reinterpret_cast<float2 *>(&sm.s[kh][16 * hg + g + 8 * r][8 * nt + 2 * t]) =
              make_float2(acc[nt][2 * r], acc[nt][2 * r + 1]);
    }
    bar_consumers(kCons);
    if (!dead) {
      // ---- online softmax, 4 threads per head
      float z[8], sg[8], mx = -INFINITY;
      const float qf = sm.qf[sh];
#pragma unroll
      for (int i = 0; i < 8; i += 4) {
        const float4 s0 = *reinterpret_cast<const float4 *>(&sm.s[0][sh][8 * sq + i]);
        const float4 s1 = *reinterpret_cast<const float4 *>(&sm.s[1][sh][8 * sq + i]);
        const float4 g4 = *reinterpret_cast<const float4 *>(&sm.sig[st][8 * sq + i]);
        z[i] = s0.x + s1.x;
        z[i + 1] = s0.y + s1.y;
        z[i + 2] = s0.z + s1.z;
        z[i + 3] = s0.w + s1.w;
        sg[i] = g4.x;
        sg[i + 1] = g4.y;
        sg[i + 2] = g4.z;
        sg[i + 3] = g4.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        z[i] = sg[i] > 0.0f ? z[i] * qf * sg[i] : -INFINITY;
        mx = fmaxf(mx, z[i]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      // a segment's first chunk (m_run = -inf) rescales O by 0: it drops the
      // previous segment's O, already written out (O is 0 before the first one)
      const float alpha = m_run == -INFINITY ? 0.0f : exp2f(m_run - m_new);
      float sum = 0.0f;
      uint32_t pw[4];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const float p0 = m_new == -INFINITY ? 0.0f : exp2f(z[i] - m_new);
        const float p1 = m_new == -INFINITY ? 0.0f : exp2f(z[i + 1] - m_new);
        sum += p0 + p1;
        __half2 h2 = __floats2half2_rn(p0 * sg[i], p1 * sg[i + 1]);
        pw[i / 2] = *reinterpret_cast<uint32_t *>(&h2);
      }
      *reinterpret_cast<uint4 *>(&sm.p[sh][8 * sq]) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      if (sq == 0) sm.alpha[sh] = alpha;
    }
    bar_consumers(kCons);
    if (!dead) {
      // ---- O = O * alpha + P V over dims d0..
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const float a0 = sm.alpha[16 * mt + g], a1 = sm.alpha[16 * mt + g + 8];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          o[mt][nt][0] *= a0;
          o[mt][nt][1] *= a0;
          o[mt][nt][2] *= a1;
          o[mt][nt][3] *= a1;
        }
      }
#pragma unroll
      for (int ks = 0; ks < kE / 16; ++ks) {
        uint32_t af[kMT][4];
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt)
          ldsm_x4(smem_u32(&sm.p[16 * mt + (lane & 15)][16 * ks + (lane >> 4) * 8]), af[mt][0], af[mt][1], af[mt][2],
                  af[mt][3]);
        const uint32_t vb = smem_u32(&sm.kv[st][16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8][d0 + (lane >> 4) * 8]);
#pragma unroll
        for (int nt = 0; nt < kNT; nt += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + nt * 16, b0, b1, b2, b3);
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt) {
            mma_f16(o[mt][nt], af[mt], b0, b1);
            mma_f16(o[mt][nt + 1], af[mt], b2, b3);
          }
        }
      }
    }
    tc::mbar_arrive(&sm.empty[st]);
    const int seg = sm.seg_end[c];
    if (n_seg > 1 && seg >= 0) {
      // ---- the segment ends: its unnormalised O and (m, l) go to its slot of
      // the workspace, and the next segment starts from nothing (with m = -inf
      // its first chunk rescales O by 0).  A wait that ran out in any consumer
      // warp voids the segment (the error bit is raised).
      const int alive = bar_consumers_and(kCons, dead ? 0 : 1);
      float *mine = part_ws + (static_cast<size_t>(row * gridDim.z + blockIdx.z) * n_seg + seg) * part_floats<HP>();
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int hl = 16 * mt + g + 8 * r;
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt)
            *reinterpret_cast<float2 *>(mine + hl * kLat + d0 + 8 * nt + 2 * t) =
                make_float2(o[mt][nt][2 * r], o[mt][nt][2 * r + 1]);
        }
      if (sq == 0)
        *reinterpret_cast<float2 *>(mine + HP * kLat + 2 * sh) =
            alive ? make_float2(m_run, l_run) : make_float2(-INFINITY, 0.0f);
      m_run = -INFINITY;
      l_run = 0.0f;
    }
  }

  if (n_seg > 1) {
    // ---- every segment's partial is in the workspace: after the cluster
    // barrier (release / acquire at cluster scope) CTA `cta` merges heads cta,
    // cta + G, ... over all segments
    cluster_sync();
    const float *part_row = part_ws + static_cast<size_t>(row * gridDim.z + blockIdx.z) * n_seg * part_floats<HP>();
    if (n_seg <= 4)
      merge_heads<4, 2, HP>(a, part_row, row, hbase, nh, cta, n_cta, n_seg, warp, kCons / 32, lane);
    else
      merge_heads<kMaxSeg, 1, HP>(a, part_row, row, hbase, nh, cta, n_cta, n_seg, warp, kCons / 32, lane);
    return;
  }

  // ---- one segment: normalise in registers
  if (sq == 0) {
    sm.fin[sh][0] = m_run;
    sm.fin[sh][1] = l_run;
  }
  // a wait that ran out in any consumer warp: the CTA's result is void (the
  // error bit is raised); it still takes part in every barrier below
  const int alive = bar_consumers_and(kCons, dead ? 0 : 1);
  if (!alive) return;
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int hl = 16 * mt + g + 8 * r;
      if (hl >= nh) continue;
      const int h = hbase + hl;
      float m = sm.fin[hl][0], l = sm.fin[hl][1], f = 1.0f;
      if (a.sink) {
        const float s2 = a.sink[h] * kLog2e;
        const float mf = fmaxf(m, s2);
        f = (m == -INFINITY) ? 0.0f : exp2f(m - mf);
        l = l * f + exp2f(s2 - mf);
        m = mf;
      }
      const float inv = l > 0.0f ? f / l : 0.0f;
      float *out = a.out + (static_cast<size_t>(row) * a.heads + h) * kLat + d0;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
        *reinterpret_cast<float2 *>(out + 8 * nt + 2 * t) =
            make_float2(o[mt][nt][2 * r] * inv, o[mt][nt][2 * r + 1] * inv);
      if (warp == 0 && t == 0) a.lse[static_cast<size_t>(row) * a.heads + h] = l > 0.0f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
}

// ============================================================================ tensor-core kernel
// One-segment rows (the chunked prefill): one CTA = one query row and 64 heads,
// the row's chunks in order, with both contractions on the 5th-generation tensor
// cores:
// tcgen05.mma kind::f16, fp16 operands in shared memory, fp32 accumulators in
// tensor memory (TMEM).
//   S = Q K^T        M = 64 heads, N = 32 entries, K = 576 (36 MMAs); head h's
//                    row of S sits in TMEM lane 32 (h / 16) + h % 16
//   O^T += V^T P^T   four blocks of M = 128 latent dims x N = 64 heads, K = the
//                    chunk's 32 entries (the fp16 tile read MN-major); O^T of
//                    block b in TMEM columns 64 + 64 b, dim 128 b + lane
// Roles (384 threads):
//   warps 0-3  query to fp16 (once); per chunk the softmax (lanes 0-15 of warp
//              w: heads 16w .. 16w + 15) and, after the last chunk, the
//              normalised O read-out of blocks 0, 1 (every thread one TMEM
//              lane; the producer warps read blocks 2, 3); P (fp16, times the
//              entry's 2^sigma) goes to shared memory as the B operand.  A
//              head's reference max moves only when some 2^sigma-weighted logit
//              of the chunk would exceed it by more than 2^kSlack; O^T's column
//              of that head is then rescaled in TMEM before the chunk's PV
//   warps 4-7  producers, as in k_attn, into a three-stage tile in the operand
//              layout (core matrices of 8 entries x 8 dims)
//   warp 8     one thread issues every MMA: PV of chunk c, then S of chunk
//              c + 2 (its tile and its S buffer are free by then), so the
//              tensor core computes S ahead of the softmax
//   warps 8-11 with warps 0-3, the query to fp16 (eight heads per warp)
// Every wait is bounded (CSA2_DEVERR_TIMEOUT if one runs out).
constexpr int kTcHeads = 64;
constexpr int kTcStages = 3;
constexpr int kTcMmaWarp = 8;
constexpr int kTcThreads = 32 * 12;
constexpr int kQBytes = kTcHeads * kDqk * 2;   // 73,728
constexpr int kTileBytes = kE * kDqk * 2;      // 36,864
constexpr int kPBytes = kTcHeads * kE * 2;     // 4,096
constexpr float kSlack = 15.0f;                // P * 2^sigma stays below 2^16 (fp16)
constexpr uint32_t kTcCols = 512;              // S[2]: columns 0..63; O^T block b: 64 + 64 b

// Operand layouts (no swizzle; core matrices of 8 rows x 16 bytes).
//   Q (head h, dim d): A of S, K-major                     LBO 1024, SBO 128
__device__ __forceinline__ uint32_t q_off(int h, int d) {
  return static_cast<uint32_t>((d >> 3) * 1024 + (h >> 3) * 128 + (h & 7) * 16 + (d & 7) * 2);
}
//   tile (entry e, dim d): B of S, K-major (N = e)         LBO 512, SBO 128
//                          A of O^T, MN-major (M = d)       LBO 128, SBO 512
__device__ __forceinline__ uint32_t t_off(int e, int d) {
  return static_cast<uint32_t>((d >> 3) * 512 + (e >> 3) * 128 + (e & 7) * 16 + (d & 7) * 2);
}
//   P (head h, entry e): B of O^T, K-major (N = h)          LBO 1024, SBO 128
__device__ __forceinline__ uint32_t p_off(int h, int e) {
  return static_cast<uint32_t>((e >> 3) * 1024 + (h >> 3) * 128 + (h & 7) * 16 + (e & 7) * 2);
}
// kind::f16 instruction descriptor: fp16 x fp16 -> fp32; a_mn marks an MN-major A
__host__ __device__ __forceinline__ uint32_t idesc_f16(int m, int n, int a_mn) {
  uint32_t d = 1u << 4;  // D format fp32; A and B fp16
  d |= static_cast<uint32_t>(a_mn & 1) << 15;
  d |= static_cast<uint32_t>((n >> 3) & 0x3F) << 17;
  d |= static_cast<uint32_t>((m >> 4) & 0x1F) << 24;
  return d;
}
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// named barrier over the softmax warps returning the OR of v
__device__ __forceinline__ int bar_sm_or(int v) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, 2, 128, p;\n selp.s32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v)
      : "memory");
  return r;
}
__device__ __forceinline__ int bar_sm_and(int v) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.and.pred q, 2, 128, p;\n selp.s32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v)
      : "memory");
  return r;
}

// Read-out of O^T blocks [b0, b1) of one TMEM lane quarter into O rows:
// dst[h * 512 + 128 b + d] = O^T[d][h] * fin[h] for the heads h < nh; the warp
// reads lanes lane_base .. + 31 (dims 128 b + d_lane), four 16-column loads in
// flight, then stores each head's 32 dims as one coalesced 128-byte row piece.
__device__ __forceinline__ void read_out(uint32_t tmem, uint32_t lane_base, int d_lane, int b0, int b1, float *dst,
                                         const float *fin, int nh) {
#pragma unroll 1
  for (int b = b0; b < b1; ++b) {
    uint32_t r[4][16];
#pragma unroll
    for (int q = 0; q < 4; ++q) tc::tmem_ld_32x32b_x16(tmem + lane_base + 64 + 64 * b + 16 * q, r[q]);
#pragma unroll
    for (int q = 0; q < 4; ++q) tc::tmem_ld_wait_x16(r[q]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (16 * q + i < nh) dst[(16 * q + i) * kLat + 128 * b + d_lane] = __uint_as_float(r[q][i]) * fin[16 * q + i];
  }
}
__device__ __forceinline__ void bar_ro() { asm volatile("bar.sync 3, 256;\n" ::: "memory"); }

struct __align__(1024) TcAttnSmem {
  uint8_t q[kQBytes];
  uint8_t tile[kTcStages][kTileBytes];
  uint8_t p[2][kPBytes];
  __align__(16) float qf[kTcHeads];    // logit factor of head h: 2^e_h * sm_scale * log2(e)
  __align__(16) float alpha[kTcHeads]; // this chunk's rescale of head h's O^T column (1: none)
  __align__(16) float fin[kTcHeads];   // output factor of head h (one-segment rows)
  __align__(16) float sig[kTcStages][kE];  // 2^sigma_j of entry j of a stage (read as float4); 0 = empty entry
  __align__(16) float sgm[kTcStages][kE];  // sigma_j (-inf for an empty entry)
  int32_t sel[kMaxChunks][kE];  // selected index of entry e of chunk i (-1: none)
  uint32_t tmem;
  int ro_alive;  // the row's result is valid (no wait ran out)
  __align__(8) uint64_t full[kTcStages];
  __align__(8) uint64_t empty[kTcStages];
  __align__(8) uint64_t s_full[2];
  __align__(8) uint64_t p_full[2];
  __align__(8) uint64_t pv_done[2];
  __align__(8) uint64_t q_ready;
};

// grid (rows, head blocks of 64)
__global__ void __launch_bounds__(kTcThreads, 1) k_attn_tc(AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TcAttnSmem &sm = *reinterpret_cast<TcAttnSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x, hbase = blockIdx.y * kTcHeads;
  const int nh = min(kTcHeads, a.heads - hbase);
  float *out_rows = a.out + (static_cast<size_t>(row) * a.heads + hbase) * kLat;  // O[h][d] of this CTA's heads
  const int seq = a.cache_seq < 0 ? row : a.cache_seq;
  const int kpad = (a.k + kE - 1) / kE * kE;
  const int total_chunks = (kpad + kWin) / kE;

  if (warp == kTcMmaWarp) {
    tc::tmem_alloc(&sm.tmem, kTcCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      tc::mbar_init(&sm.full[i], kProdThreads);
      tc::mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm.s_full[i], 1);
      tc::mbar_init(&sm.p_full[i], 4);
      tc::mbar_init(&sm.pv_done[i], 1);
    }
    tc::mbar_init(&sm.q_ready, 8);
    tc::fence_mbar_init();
  }
  // a programmatic dependent of the previous kernel: nothing in memory is read
  // before that grid is complete
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const int nchunks = total_chunks;  // the row's chunks, in order
  const int64_t qpos = a.q_pos[row];
  const int64_t T = qpos / a.ratio;
  const int64_t ntok = a.n_tokens[seq];
  const int64_t lin_base = a.lin_base ? *a.lin_base : INT64_MAX;

  // the query to fp16 with a power-of-two scale per head (|q * 2^-e| < 2^15):
  // warps 0-3 and 8-11 convert eight heads each (qw, qw + 8, ...), every raw
  // value of the eight requested before any is used (one round trip)
  if (warp < 4 || warp >= kTcMmaWarp) {
    constexpr int kQW = kTcHeads / 8, kQP = kDqk / 2 / 32;
    const int qw = warp < 4 ? warp : warp - 4;
    uint32_t raw[kQW][kQP];
#pragma unroll
    for (int j = 0; j < kQW; ++j) {
      const int h = qw + 8 * j;
      const uint32_t *gq =
          reinterpret_cast<const uint32_t *>(a.q + (static_cast<size_t>(row) * a.heads + hbase + h) * kDqk);
#pragma unroll
      for (int i = 0; i < kQP; ++i) raw[j][i] = h < nh ? __ldg(gq + lane + 32 * i) : 0u;
    }
    float amax[kQW];
#pragma unroll
    for (int j = 0; j < kQW; ++j) {
      amax[j] = 0.0f;
#pragma unroll
      for (int i = 0; i < kQP; ++i)
        amax[j] = fmaxf(amax[j], fmaxf(fabsf(__uint_as_float(raw[j][i] << 16)),
                                       fabsf(__uint_as_float(raw[j][i] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1)
#pragma unroll
      for (int j = 0; j < kQW; ++j) amax[j] = fmaxf(amax[j], __shfl_xor_sync(0xffffffffu, amax[j], o));
#pragma unroll
    for (int j = 0; j < kQW; ++j) {
      const int h = qw + 8 * j;
      int ex = amax[j] > 0.0f ? floor_log2f(amax[j]) - 14 : 0;
      ex = max(ex, -110);
      const float inv = pow2f(-ex);
#pragma unroll
      for (int i = 0; i < kQP; ++i) {
        __half2 t2 = __floats2half2_rn(__fmul_rn(__uint_as_float(raw[j][i] << 16), inv),
                                       __fmul_rn(__uint_as_float(raw[j][i] & 0xFFFF0000u), inv));
        *reinterpret_cast<__half2 *>(sm.q + q_off(h, 2 * (lane + 32 * i))) = t2;
      }
      if (lane == 0) sm.qf[h] = h < nh ? pow2f(ex) * a.sm_scale * kLog2e : 0.0f;
    }
    tc::fence_proxy_async_smem();  // Q is read by the tensor cores
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&sm.q_ready);
  }

  if (warp >= 4 && warp < 8) {
    // ================================================================ producers
    const int pt = tid - 128;
    const int e = pt >> 2, q4 = pt & 3;
    const uint32_t qmask = 0xFu << (lane & ~3);
    const int32_t *idx_row = a.idx + static_cast<size_t>(row) * a.k;
    // the selected indices of every chunk of this CTA, loaded once (one round
    // trip) into shared memory: a chunk's record address is then known at once
    for (int i = pt; i < nchunks * kE; i += kProdThreads) {
      const int j = i;  // entry j of the row's list: chunk j / 32
      sm.sel[i / kE][i % kE] = j < a.k ? idx_row[j] : -1;
    }
    asm volatile("bar.sync 4, %0;\n" ::"r"(kProdThreads) : "memory");
    auto sel_of = [&](int i) -> int32_t { return sm.sel[i][e]; };
    // two chunks in flight: chunk c is dequantised from one record buffer while
    // chunk c + 1's loads land in the other; chunk c + 2's are then issued into
    // the first (no register copies, so no wait on a load before its use)
    const bool fp8 = a.entry_format == CSA2_ENTRY_FP8;
    struct Rec {
      int kind;
      int64_t src;
      Fp4Raw raw;
    };
    auto fetch = [&](int c, Rec &r) {  // chunk c's record: FP4 into registers, other kinds into L2
      r.kind = entry_kind(a, seq, c * kE + e, kpad, sel_of(c), qpos, T, ntok, lin_base, r.src);
      if (r.kind == 1 && !fp8) load_fp4_early(a, r.src, q4, r.raw);
      else prefetch_entry(a, r.kind, r.src, q4, fp8);
    };
    bool dead = false;
    auto produce = [&](int c, Rec &r) {
      const int ts = c % kTcStages;
      if (c >= kTcStages && !dead) dead = !wait_warp(&sm.empty[ts], ((c / kTcStages) - 1) & 1, a.err);
      if (!dead) {
        uint8_t *tile = sm.tile[ts];
        const float sig = dequant_entry(a, r.kind, r.src, r.raw, q4, qmask, fp8, [&](int u, uint4 lo, uint4 hi) {
          *reinterpret_cast<uint4 *>(tile + t_off(e, 16 * u)) = lo;
          *reinterpret_cast<uint4 *>(tile + t_off(e, 16 * u + 8)) = hi;
        });
        if (q4 == 0) {
          sm.sig[ts][e] = sig;
          sm.sgm[ts][e] = sig > 0.0f ? static_cast<float>(floor_log2f(sig)) : -INFINITY;
        }
      }
      tc::fence_proxy_async_smem();  // the tile is read by the tensor cores
      tc::mbar_arrive(&sm.full[ts]);
      if (c + 2 < nchunks) fetch(c + 2, r);
    };
    Rec ra, rb;
    if (nchunks > 0) fetch(0, ra);
    if (nchunks > 1) fetch(1, rb);
    for (int c = 0; c < nchunks; c += 2) {
      produce(c, ra);
      if (c + 1 < nchunks) produce(c + 1, rb);
    }
    if (nchunks > 0) {
      // blocks 2, 3 of the last segment's O^T (warp 4 + w reads TMEM lanes 32 w ..)
      bar_ro();
      tc::tc_fence_after();
      if (sm.ro_alive)
        read_out(tmem, static_cast<uint32_t>(32 * (warp - 4)) << 16, 32 * (warp - 4) + lane, 2, 4, out_rows, sm.fin, nh);
      tc::tc_fence_before();
    }
  } else if (warp == kTcMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_f16(64, kE, 0), idO = idesc_f16(128, kTcHeads, 1);
      const uint32_t qa = tc::smem_addr(sm.q);
      bool dead = !tc::mbar_wait_bounded(&sm.q_ready, 0, kWaitIters);
      auto issue_qk = [&](int c) {
        const int ts = c % kTcStages, sb = c & 1;
        if (dead || !tc::mbar_wait_bounded(&sm.full[ts], (c / kTcStages) & 1, kWaitIters)) {
          dead = true;
          return;
        }
        tc::tc_fence_after();
        const uint32_t ta = tc::smem_addr(sm.tile[ts]);
#pragma unroll 4
        for (int kk = 0; kk < kDqk / 16; ++kk)
          mma_f16_ss(tmem + 32 * sb, tc::smem_desc_noswizzle(qa + kk * 2048, 1024, 128),
                     tc::smem_desc_noswizzle(ta + kk * 1024, 512, 128), idS, kk > 0 ? 1u : 0u);
        tc::mma_commit(&sm.s_full[sb]);
      };
      if (nchunks > 0) issue_qk(0);
      if (nchunks > 1) issue_qk(1);
      for (int c = 0; c < nchunks && !dead; ++c) {
        const int ts = c % kTcStages, sb = c & 1;
        if (!tc::mbar_wait_bounded(&sm.p_full[sb], (c >> 1) & 1, kWaitIters)) {
          dead = true;
          break;
        }
        const bool first = c == 0;
        tc::tc_fence_after();
        const uint32_t ta = tc::smem_addr(sm.tile[ts]), pa = tc::smem_addr(sm.p[sb]);
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            mma_f16_ss(tmem + 64 + 64 * b, tc::smem_desc_noswizzle(ta + 8192 * b + 256 * ks, 128, 512),
                       tc::smem_desc_noswizzle(pa + 2048 * ks, 1024, 128), idO, (first && ks == 0) ? 0u : 1u);
        tc::mma_commit(&sm.empty[ts]);
        tc::mma_commit(&sm.pv_done[sb]);
        if (c + 2 < nchunks) issue_qk(c + 2);
      }
      if (dead) raise_err(a.err, CSA2_DEVERR_TIMEOUT);
    }
  } else if (warp < 4) {
    // ================================================================ softmax / O^T (warps 0-3)
    const bool head_thread = lane < 16;
    const int h = 16 * warp + lane;  // this thread's head (head_thread)
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    float m_ref = -INFINITY, l_run = 0.0f;
    bool dead = !wait_warp(&sm.q_ready, 0, a.err);  // qf of every head written
    const float qf = head_thread ? sm.qf[h] : 0.0f;
    for (int c = 0; c < nchunks; ++c) {
      const int ts = c % kTcStages, sb = c & 1;
      // P buffer sb is free once PV of chunk c - 2 is complete
      if (c >= 2 && !dead) dead = !wait_warp(&sm.pv_done[sb], ((c - 2) >> 1) & 1, a.err);
      if (!dead) dead = !wait_warp(&sm.s_full[sb], (c >> 1) & 1, a.err);
      tc::tc_fence_after();
      uint32_t sv[32];
      tc::tmem_ld_32x32b_x16(tmem + lane_base + 32 * sb, sv);
      tc::tmem_ld_32x32b_x16(tmem + lane_base + 32 * sb + 16, sv + 16);
      tc::tmem_ld_wait_x16(sv);
      tc::tmem_ld_wait_x16(sv + 16);
      int moved = 0;
      if (head_thread && !dead) {
        // logits z_j = s_j qf 2^sigma_j (in place of s_j), and the largest
        // weighted logit z_j + sigma_j, which bounds P_j 2^sigma_j
        float my = -INFINITY;
#pragma unroll
        for (int j = 0; j < kE; j += 4) {
          const float4 g4 = *reinterpret_cast<const float4 *>(&sm.sig[ts][j]);
          const float4 s4 = *reinterpret_cast<const float4 *>(&sm.sgm[ts][j]);
          const float g[4] = {g4.x, g4.y, g4.z, g4.w}, sg[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float zz = g[i] > 0.0f ? __uint_as_float(sv[j + i]) * qf * g[i] : -INFINITY;
            sv[j + i] = __float_as_uint(zz);
            my = fmaxf(my, zz + sg[i]);
          }
        }
        float m_new = m_ref, alpha = 1.0f;
        if (my != -INFINITY) {
          if (m_ref == -INFINITY) {
            m_new = my;  // this head's first entries: O^T's column is still zero
          } else if (my > m_ref + kSlack) {
            m_new = my;
            alpha = exp2f(m_ref - m_new);
            moved = 1;
          }
        }
        float sum = 0.0f;
        uint8_t *pb = sm.p[sb];
        const float mz = m_new == -INFINITY ? 0.0f : m_new;  // exp2(-inf - mz) = 0 for every empty entry
#pragma unroll
        for (int j = 0; j < kE; j += 8) {
          const float4 ga = *reinterpret_cast<const float4 *>(&sm.sig[ts][j]);
          const float4 gb = *reinterpret_cast<const float4 *>(&sm.sig[ts][j + 4]);
          const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            const float p0 = exp2f(__uint_as_float(sv[j + i]) - mz);
            const float p1 = exp2f(__uint_as_float(sv[j + i + 1]) - mz);
            sum += p0 + p1;
            __half2 h2 = __floats2half2_rn(p0 * g[i], p1 * g[i + 1]);
            w[i / 2] = *reinterpret_cast<uint32_t *>(&h2);
          }
          *reinterpret_cast<uint4 *>(pb + p_off(h, j)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        l_run = l_run * alpha + sum;
        m_ref = m_new;
        sm.alpha[h] = alpha;
      }
      // some head moved its reference: its O^T column is rescaled once PV of
      // chunk c - 1 is complete (the first chunk starts O^T instead)
      if (bar_sm_or(moved) && c > 0) {
        if (!dead) dead = !wait_warp(&sm.pv_done[sb ^ 1], ((c - 1) >> 1) & 1, a.err);
        tc::tc_fence_after();
#pragma unroll 1
        for (int b = 0; b < 4; ++b)
#pragma unroll 1
          for (int h0 = 0; h0 < kTcHeads; h0 += 16) {
            uint32_t r[16];
            const uint32_t ta = tmem + lane_base + 64 + 64 * b + h0;
            tc::tmem_ld_32x32b_x16(ta, r);
            tc::tmem_ld_wait_x16(r);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * sm.alpha[h0 + i]);
            tmem_st_32x32b_x16(ta, r);
          }
        asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
      }
      tc::fence_proxy_async_smem();  // P is read by the tensor cores
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.p_full[sb]);
      if (c == nchunks - 1) {
        // ---- the last chunk: O^T is complete once its PV is; normalise (with
        // the sink) and write the row's output, blocks 0, 1 here and 2, 3 by the
        // producer warps
        if (!dead) dead = !wait_warp(&sm.pv_done[sb], (c >> 1) & 1, a.err);
        tc::tc_fence_after();
        const int alive = bar_sm_and(dead ? 0 : 1);
        if (head_thread) {
          float m = m_ref, l = l_run, f = 1.0f;
          if (h < nh && a.sink) {
            const float s2 = a.sink[hbase + h] * kLog2e;
            const float mf = fmaxf(m, s2);
            f = (m == -INFINITY) ? 0.0f : exp2f(m - mf);
            l = l * f + exp2f(s2 - mf);
            m = mf;
          }
          sm.fin[h] = l > 0.0f ? f / l : 0.0f;
          if (h < nh && alive)
            a.lse[static_cast<size_t>(row) * a.heads + hbase + h] = l > 0.0f ? (m + log2f(l)) * kLn2 : -INFINITY;
        }
        if (tid == 0) sm.ro_alive = alive;
        bar_ro();  // fin and ro_alive written; the producer warps join here
        if (alive) read_out(tmem, lane_base, 32 * warp + lane, 0, 2, out_rows, sm.fin, nh);
        tc::tc_fence_before();
      }
    }
  }

  // ---- teardown of the tensor memory
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTcCols);
  }
}

cudaError_t launch_tc(const AttnArgs &a, cudaStream_t st) {
  const int smem = static_cast<int>(sizeof(TcAttnSmem)) + 1024;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(k_attn_tc), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.rows, (a.heads + kTcHeads - 1) / kTcHeads);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_attn_tc, a);
}

int head_blocks(int heads, int hp) { return (heads + hp - 1) / hp; }

// Launch shape: G CTAs per (row, head block), one cluster, and hp heads per CTA.
// The segments of a row are fixed; G only spreads them, and a head's arithmetic
// does not depend on the head block it is in, so neither choice changes a bit.
// G grows first (up to one CTA per segment) while the grid fits one wave of one
// CTA per SM; then, for small batches, the heads are split into blocks of 32 or
// 16 (each CTA then dequantises the row's entries for fewer heads).
struct AttnShape {
  int n_cta, hp;
};
AttnShape choose_shape(int rows, int heads, int n_seg) {
  const int sms = device_sm_count();
  AttnShape sh{1, heads <= 16 ? 16 : heads <= 32 ? 32 : kHeadBlock};
  const int ctas = rows * head_blocks(heads, sh.hp);
  sh.n_cta = sms / ctas;
  if (sh.n_cta > n_seg) sh.n_cta = n_seg;
  if (sh.n_cta < 1) sh.n_cta = 1;
  while (sh.hp > 16 && sh.n_cta == n_seg && rows * sh.n_cta * head_blocks(heads, sh.hp / 2) <= sms) sh.hp /= 2;
  return sh;
}

template <int HP>
cudaError_t launch_hp(const AttnArgs &a, int n_cta, int n_seg, float *part, cudaStream_t st) {
  const int smem = static_cast<int>(sizeof(AttnSmem<HP>));
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(k_attn<HP>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_cta, a.rows, head_blocks(a.heads, HP));
  cfg.blockDim = dim3(HP * 4 + kProdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = n_cta;  // the row's CTAs of one head block: one cluster
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_attn<HP>, a, n_cta, n_seg, part);
}

}  // namespace

// Segments of a decode row's entry list: fixed by k and the window alone (never
// by the batch), four, or fewer when the list has fewer 32-entry chunks.
int attn_segments(int k) {
  const int chunks = ((k + kE - 1) / kE * kE + kWin) / kE;
  return chunks < kSegments ? chunks : kSegments;
}

// Workspace: the partial (O, m, l) of every segment of every (row, head) when a
// row has more than one segment (sized for 64-head blocks, the largest: a
// smaller block never needs more).
size_t attn_workspace_bytes(int rows, int heads, int n_seg) {
  if (n_seg <= 1) return 256;
  return static_cast<size_t>(rows) * head_blocks(heads, kHeadBlock) * n_seg * part_floats<kHeadBlock>() *
             sizeof(float) +
         256;
}

cudaError_t launch_attn(const AttnArgs &a0, int n_seg, void *ws, size_t ws_bytes, cudaStream_t st) {
  if (a0.rows <= 0) return cudaSuccess;
  if (n_seg < 1 || n_seg > kMaxSeg) return cudaErrorInvalidValue;
  const AttnShape sh = choose_shape(a0.rows, a0.heads, n_seg);
  if (n_seg > 1 && (ws == nullptr || ws_bytes + 256 < attn_workspace_bytes(a0.rows, a0.heads, n_seg) ||
                    reinterpret_cast<uintptr_t>(ws) % 16 != 0))
    return cudaErrorInvalidValue;
  float *part = static_cast<float *>(ws);
  // one-segment rows (the chunked prefill: a query's whole entry list in one
  // CTA) on the tensor-core kernel; decode rows on the mma.sync kernel, whose
  // O stays in registers (the segments' read-out and merge cost more from TMEM
  // than the faster contractions save on a 5-chunk segment)
  if (n_seg == 1) return launch_tc(a0, st);
  if (sh.hp == 16) return launch_hp<16>(a0, sh.n_cta, n_seg, part, st);
  if (sh.hp == 32) return launch_hp<32>(a0, sh.n_cta, n_seg, part, st);
  return launch_hp<64>(a0, sh.n_cta, n_seg, part, st);
}

}  // namespace csa2
