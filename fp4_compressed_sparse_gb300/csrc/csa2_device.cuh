// csa2_device.cuh -- device-side number formats, quantisers and launch helpers
// shared by the libcsa2 kernels (sm_103a).
//
// Formats ([P1] "DeepSeek V4.1 Flash 아키텍처 분석", §"890 bytes/token은 어떻게
// 나오는가"): main KV = E2M1 codes with one E4M3 scale per 16 values; indexer
// key = MXFP4 (E2M1 with one E8M0 scale per 32); window KV in 8 bits (MXFP8:
// E4M3 with one E8M0 scale per 32) or bf16.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa2.h"

namespace csa2 {

constexpr int kLat = CSA2_D_LATENT;  // 512
constexpr int kRope = CSA2_D_ROPE;   // 64
constexpr int kDqk = CSA2_D_QK;      // 576
constexpr int kDi = CSA2_D_INDEX;    // 128
constexpr int kDcmp = CSA2_D_CMP;    // 704
constexpr int kWin = CSA2_WINDOW;    // 128
constexpr int kSwaScaleStride = 32;  // bytes per window slot in swa_scales (18 used)

// Indexer-key planes are stored tile-major, in the operand layout the
// block-scaled tensor-core MMA reads, so that a 128-entry tile is one
// contiguous 8 KB code block plus one 512 B scale block:
//   codes: tile*8192 + chunk*2048 + m*16 + byte   (m = entry % 128, chunk = 16-byte
//          piece = one 32-value MXFP4 block of the 128-dim key)
//   scales: tile*512 + 16*(m % 32) + 4*(m / 32) + block
constexpr int kIdxTile = 128;
constexpr int kIdxTileCodeBytes = 8192;
constexpr int kIdxTileScaleBytes = 512;
__host__ __device__ __forceinline__ int64_t idx_tiles(int64_t capacity) { return (capacity + kIdxTile - 1) / kIdxTile; }
// byte offsets of block `chunk` of row m (0..127) of physical tile `tile`
__host__ __device__ __forceinline__ size_t idx_code_at(int64_t tile, int m, int chunk) {
  return static_cast<size_t>(tile) * kIdxTileCodeBytes + chunk * 2048 + m * 16;
}
__host__ __device__ __forceinline__ size_t idx_scale_at(int64_t tile, int m) {
  return static_cast<size_t>(tile) * kIdxTileScaleBytes + 16 * (m % 32) + 4 * (m / 32);
}

// ---------------------------------------------------------------- entry addressing
// Where entry e of sequence b lives: the dense layout ([batch][capacity], each
// sequence's entries contiguous, its indexer tiles padded per sequence) or the
// paged one (a block table maps page e / page of sequence b to a physical page
// of `page` entries, a multiple of 128).
struct EntryMap {
  const int32_t *bt;  // [batch][max_pages], or nullptr: dense
  int32_t page, max_pages, n_pages;
  int64_t cap;        // entries per sequence
};
__host__ __device__ __forceinline__ EntryMap entry_map(const csa2_cache &c) {
  return EntryMap{c.block_table, c.page_entries, c.max_pages, c.n_pages, c.capacity};
}
// physical entry of (b, e) for the 288 B / 36 B planes; -1 for a page id outside the pool
__host__ __device__ __forceinline__ int64_t phys_entry(const EntryMap &m, int b, int64_t e) {
  if (m.bt == nullptr) return static_cast<int64_t>(b) * m.cap + e;
  const int32_t pg = m.bt[static_cast<int64_t>(b) * m.max_pages + e / m.page];
  if (pg < 0 || pg >= m.n_pages) return -1;
  return static_cast<int64_t>(pg) * m.page + e % m.page;
}
// physical 128-entry tile of tile t of sequence b for the indexer planes; -1 as above
__host__ __device__ __forceinline__ int64_t phys_tile(const EntryMap &m, int b, int64_t t) {
  if (m.bt == nullptr) return static_cast<int64_t>(b) * idx_tiles(m.cap) + t;
  const int tpp = m.page / kIdxTile;
  const int32_t pg = m.bt[static_cast<int64_t>(b) * m.max_pages + t / tpp];
  if (pg < 0 || pg >= m.n_pages) return -1;
  return static_cast<int64_t>(pg) * tpp + t % tpp;
}

// ---------------------------------------------------------------- error word
__device__ __forceinline__ void raise_err(int32_t *err, uint32_t bit) {
  if (err) atomicOr(reinterpret_cast<unsigned int *>(err), bit);
}

// ---------------------------------------------------------------- powers of two
// 2^e as fp32 for e in [-149, 127] (exact; subnormal below -126).
__device__ __forceinline__ float pow2f(int e) {
  if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  return __uint_as_float(1u << (e + 149));
}

// floor(log2(a)) of a finite a > 0, from the bit pattern.
__device__ __forceinline__ int floor_log2f(float a) {
  uint32_t u = __float_as_uint(a);
  int ex = static_cast<int>((u >> 23) & 0xFF);
  if (ex != 0) return ex - 127;
  return (31 - __clz(static_cast<int>(u & 0x7FFFFF))) - 149;  // subnormal
}

// ---------------------------------------------------------------- E2M1
// Nearest E2M1 code of y (ties to the even code, saturating at 6); the sign bit
// is y's sign bit.  Decision thresholds are the midpoints of the grid
// {0, .5, 1, 1.5, 2, 3, 4, 6}; at a midpoint the even code wins.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  float a = fabsf(y);
  uint32_t c = (a <= 0.25f) ? 0u
             : (a < 0.75f)  ? 1u
             : (a <= 1.25f) ? 2u
             : (a < 1.75f)  ? 3u
             : (a <= 2.5f)  ? 4u
             : (a < 3.5f)   ? 5u
             : (a <= 5.0f)  ? 6u
                            : 7u;
  return c | ((__float_as_uint(y) >> 28) & 8u);
}

// Value of an E2M1 code, times 2 (an exact small integer).
// code = s|e1 e0|m: 2*value = m for e == 0, else (2 + m) << (e - 1).
__device__ __forceinline__ int e2m1_twice(uint32_t c) {
  int e = static_cast<int>((c >> 1) & 3u), m = static_cast<int>(c & 1u);
  int v = (e == 0) ? m : ((2 + m) << (e - 1));
  return (c & 8u) ? -v : v;
}

__device__ __forceinline__ float e2m1_value(uint32_t c) {
  return 0.5f * static_cast<float>(e2m1_twice(c));
}

// Four packed E2M1 codes (low 16 bits of w) -> four int8 lanes holding 2*value.
__device__ __forceinline__ uint32_t e2m1x4_twice_i8(uint32_t w) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) r |= (static_cast<uint32_t>(e2m1_twice((w >> (4 * i)) & 15u)) & 0xFFu) << (8 * i);
  return r;
}

// ---------------------------------------------------------------- E4M3 (FN)
// Round-to-nearest-even, saturating at 448; sign bit from x.
__device__ __forceinline__ uint32_t e4m3_code(float x) {
  uint32_t sign = (__float_as_uint(x) >> 24) & 0x80u;
  float a = fabsf(x);
  if (!(a <= 448.0f)) return sign | 0x7Eu;
  if (a < 0.015625f) {                       // below 2^-6: subnormal grid m * 2^-9
    uint32_t m = __float2uint_rn(a * 512.0f);  // exact scaling, RNE; m == 8 -> 0x08
    return sign | m;
  }
  uint32_t u = __float_as_uint(a);
  int e = static_cast<int>((u >> 23) & 0xFF) - 127;  // -6 .. 8
  uint32_t mant = u & 0x7FFFFFu;
  uint32_t q = mant >> 20, rem = mant & 0xFFFFFu;
  if (rem > 0x80000u || (rem == 0x80000u && (q & 1u))) ++q;
  if (q == 8u) {
    q = 0;
    ++e;
  }
  if (e > 8 || (e == 8 && q > 6u)) return sign | 0x7Eu;
  return sign | (static_cast<uint32_t>(e + 7) << 3) | q;
}

__device__ __forceinline__ float e4m3_value(uint32_t c) {
  uint32_t e = (c >> 3) & 15u, m = c & 7u;
  float v = (e == 0) ? static_cast<float>(m) * 0.001953125f
                     : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (c & 0x80u) ? -v : v;
}

// E8M0 scale 2^(c-127), c in 0..254.
__device__ __forceinline__ float e8m0_value(uint32_t c) { return pow2f(static_cast<int>(c) - 127); }

// ---------------------------------------------------------------- group quantisers
// Group of 16 with an E4M3 scale: s = E4M3(amax/6); codes E2M1(x/s) (IEEE
// divisions); s == 0 gives all-zero codes.  Returns the 8 packed bytes.
__device__ __forceinline__ uint64_t quant_nvfp4_16(const float *x, uint32_t *scale_code) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  uint32_t sc = e4m3_code(__fdiv_rn(amax, 6.0f));
  float s = e4m3_value(sc);
  uint64_t packed = 0;
  if (s != 0.0f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) packed |= static_cast<uint64_t>(e2m1_code(__fdiv_rn(x[i], s))) << (4 * i);
  } else {
    sc = 0;
  }
  *scale_code = sc;
  return packed;
}

// MXFP4 group of 32: e = floor(log2 amax) - 2 (clamped to [-127,127]); codes
// E2M1(x * 2^-e).  Writes 16 packed bytes as 4 words.
__device__ __forceinline__ void quant_mxfp4_32(const float *x, uint32_t *words4, uint32_t *scale_code) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  if (amax == 0.0f) {
    words4[0] = words4[1] = words4[2] = words4[3] = 0;
    *scale_code = 0;
    return;
  }
  int e = floor_log2f(amax) - 2;
  e = max(-127, min(127, e));
  float inv = pow2f(-e);  // -e in [-125, 127]: a normal power of two
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) word |= e2m1_code(__fmul_rn(x[8 * w + i], inv)) << (4 * i);
    words4[w] = word;
  }
  *scale_code = static_cast<uint32_t>(e + 127);
}

// MXFP8 group of 32: e = floor(log2 amax) - 8; codes E4M3(x * 2^-e).
__device__ __forceinline__ void quant_mxfp8_32(const float *x, uint32_t *words8, uint32_t *scale_code) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  if (amax == 0.0f) {
#pragma unroll
    for (int w = 0; w < 8; ++w) words8[w] = 0;
    *scale_code = 0;
    return;
  }
  int e = floor_log2f(amax) - 8;
  e = max(-127, min(127, e));
  float inv = pow2f(-e);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) word |= e4m3_code(__fmul_rn(x[4 * w + i], inv)) << (8 * i);
    words8[w] = word;
  }
  *scale_code = static_cast<uint32_t>(e + 127);
}

// ---------------------------------------------------------------- RoPE
// Pair (x, y) at table entry (c, s): x' = fma(x, c, -(y*s)), y' = fma(y, c, x*s),
// products rounded first ([P5] §2.3.3 partial RoPE on the last 64 dims).
__device__ __forceinline__ void rope_pair(float &x, float &y, float c, float s) {
  float ys = __fmul_rn(y, s), xs = __fmul_rn(x, s);
  float nx = __fmaf_rn(x, c, -ys);
  float ny = __fmaf_rn(y, c, xs);
  x = nx;
  y = ny;
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t orderable(float f) {
  // total order on fp32 (NaN excluded by the callers); -0 and +0 map equal
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace csa2
