// csa2_encode.cuh -- warp-level encoders of one cache entry and one window token
// (RoPE, then quantise; [P4] "매개변수는 커졌는데 메모리는 4분의 1 ..."
// §"890이 맞아떨어지는 계산": quantisation after RoPE).
#pragma once

#include "csa2_device.cuh"

namespace csa2 {

// Encode entry `e` of sequence b from an fp32 row in shared memory:
// row[0:576] = main vector (RoPE dims 512..575 not yet rotated), row[576:704] = indexer key.
__device__ __forceinline__ void warp_encode_entry(const csa2_cache &c, int b, int64_t e, const float *row, const float *cs,
                                  int lane) {
  const size_t ent = static_cast<size_t>(b) * c.capacity + e;
  float x[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = row[16 * lane + i];
  uint32_t sc;
  uint64_t packed = quant_nvfp4_16(x, &sc);
  reinterpret_cast<uint2 *>(c.lat_codes + ent * 256)[lane] =
      make_uint2(static_cast<uint32_t>(packed), static_cast<uint32_t>(packed >> 32));
  c.lat_scales[ent * 32 + lane] = static_cast<uint8_t>(sc);
  if (lane < 4) {
    // RoPE group `lane`: dims 512+16*lane .. +15 = pairs 8*lane .. 8*lane+7
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int pair = 8 * lane + p;
      float a = row[kLat + 2 * pair], bb = row[kLat + 2 * pair + 1];
      rope_pair(a, bb, cs[2 * pair], cs[2 * pair + 1]);
      x[2 * p] = a;
      x[2 * p + 1] = bb;
    }
    packed = quant_nvfp4_16(x, &sc);
    reinterpret_cast<uint2 *>(c.rope_codes + ent * 32)[lane] =
        make_uint2(static_cast<uint32_t>(packed), static_cast<uint32_t>(packed >> 32));
    c.rope_scales[ent * 4 + lane] = static_cast<uint8_t>(sc);
  } else if (lane < 8) {
    const int blk = lane - 4;
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = row[kDqk + 32 * blk + i];
    uint32_t w[4];
    quant_mxfp4_32(x, w, &sc);
    const int64_t tbase = static_cast<int64_t>(b) * idx_tiles(c.capacity);
    *reinterpret_cast<uint4 *>(c.idx_codes + idx_code_off(tbase, e, blk)) = make_uint4(w[0], w[1], w[2], w[3]);
    c.idx_scales[idx_scale_off(tbase, e) + blk] = static_cast<uint8_t>(sc);
  }
}

// Encode one window token from an fp32 row (576 dims, RoPE dims unrotated) into
// codes (576 B MXFP8 or 1152 B bf16) and scales (18 B, MXFP8).
__device__ __forceinline__ void warp_encode_swa(uint8_t *codes, uint8_t *scales, int swa_dtype, const float *row,
                                const float *cs, int lane) {
  float x[32];
  if (swa_dtype == CSA2_SWA_MXFP8) {
    if (lane < 18) {
      if (lane < 16) {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = row[32 * lane + i];
      } else {
#pragma unroll
        for (int p = 0; p < 16; ++p) {
          const int pair = 16 * (lane - 16) + p;
          float a = row[kLat + 2 * pair], bb = row[kLat + 2 * pair + 1];
          rope_pair(a, bb, cs[2 * pair], cs[2 * pair + 1]);
          x[2 * p] = a;
          x[2 * p + 1] = bb;
        }
      }
      uint32_t w[8], sc;
      quant_mxfp8_32(x, w, &sc);
      uint4 *dst = reinterpret_cast<uint4 *>(codes + 32 * lane);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      scales[lane] = static_cast<uint8_t>(sc);
    }
  } else {
    __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(codes);
#pragma unroll
    for (int i = 0; i < 16; ++i) h[16 * lane + i] = __float2bfloat16_rn(row[16 * lane + i]);
    if (lane < 4) {
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const int pair = 8 * lane + p;
        float a = row[kLat + 2 * pair], bb = row[kLat + 2 * pair + 1];
        rope_pair(a, bb, cs[2 * pair], cs[2 * pair + 1]);
        h[kLat + 2 * pair] = __float2bfloat16_rn(a);
        h[kLat + 2 * pair + 1] = __float2bfloat16_rn(bb);
      }
    }
  }
}

}  // namespace csa2
