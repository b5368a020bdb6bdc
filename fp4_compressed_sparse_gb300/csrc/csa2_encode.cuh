// csa2_encode.cuh -- warp-level encoders of one cache entry and one window token
// (RoPE, then quantise; [P4] "매개변수는 커졌는데 메모리는 4분의 1 ..."
// §"890이 맞아떨어지는 계산": quantisation after RoPE).
#pragma once

#include "csa2_device.cuh"

namespace csa2 {

// Encode entry `e` of sequence b from an fp32 row in shared memory:
// row[0:576] = main vector (RoPE dims 512..575 not yet rotated), row[576:704] = indexer key.
// The cache's entry format decides the record: V4.1 FP4 (the 288 B record and
// the 36 B RoPE sidecar) or V4 (MXFP8 latent, bf16 RoPE dims).  A paged cache
// whose table names a page outside the pool gets the INDEX bit.
__device__ __forceinline__ void warp_encode_entry(const csa2_cache &c, int b, int64_t e, const float *row, const float *cs,
                                                  int lane, int32_t *err) {
  const EntryMap map = entry_map(c);
  const int64_t pe = phys_entry(map, b, e), pt = phys_tile(map, b, e / kIdxTile);
  if (pe < 0 || pt < 0) {  // a page id outside the pool: nothing written
    if (lane == 0) raise_err(err, CSA2_DEVERR_INDEX);
    return;
  }
  const size_t ent = static_cast<size_t>(pe);
  float x[32];
  uint32_t sc;
  if (c.entry_format == CSA2_ENTRY_FP8) {
    // V4 entry: latent block `lane` (32 dims) in MXFP8, RoPE dims rotated into bf16
    if (lane < 16) {
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = row[32 * lane + i];
      uint32_t w[8];
      quant_mxfp8_32(x, w, &sc);
      uint4 *dst = reinterpret_cast<uint4 *>(c.lat_codes + ent * 512 + 32 * lane);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      c.lat_scales[ent * 16 + lane] = static_cast<uint8_t>(sc);
    } else if (lane < 20) {
      __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(c.rope_codes + ent * 128);
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const int pair = 8 * (lane - 16) + p;
        float a = row[kLat + 2 * pair], bb = row[kLat + 2 * pair + 1];
        rope_pair(a, bb, cs[2 * pair], cs[2 * pair + 1]);
        h[2 * pair] = __float2bfloat16_rn(a);
        h[2 * pair + 1] = __float2bfloat16_rn(bb);
      }
    } else if (lane < 24) {
      const int blk = lane - 20;
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = row[kDqk + 32 * blk + i];
      uint32_t w[4];
      quant_mxfp4_32(x, w, &sc);
      *reinterpret_cast<uint4 *>(c.idx_codes + idx_code_at(pt, e % kIdxTile, blk)) = make_uint4(w[0], w[1], w[2], w[3]);
      c.idx_scales[idx_scale_at(pt, e % kIdxTile) + blk] = static_cast<uint8_t>(sc);
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = row[16 * lane + i];
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
    *reinterpret_cast<uint4 *>(c.idx_codes + idx_code_at(pt, e % kIdxTile, blk)) = make_uint4(w[0], w[1], w[2], w[3]);
    c.idx_scales[idx_scale_at(pt, e % kIdxTile) + blk] = static_cast<uint8_t>(sc);
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

// ---------------------------------------------------------------- block encoders
// The same encodings with a whole 256-thread block on one token: every thread
// quantises 1..4 values and group maxima are lane shuffles, so the token's
// ~1,300 values take a few dependent steps instead of one warp's long loops.
constexpr int kEncThreads = 256;

// rot[0:64] = RoPE dims of row (row[512:576]) rotated with cs; threads 0..31.
__device__ __forceinline__ void block_rope(const float *row, const float *cs, float *rot) {
  const int t = threadIdx.x;
  if (t < 32) {
    float a = row[kLat + 2 * t], bb = row[kLat + 2 * t + 1];
    rope_pair(a, bb, cs[2 * t], cs[2 * t + 1]);
    rot[2 * t] = a;
    rot[2 * t + 1] = bb;
  }
}

// The same with the table row already in rot[0:64] (cos, sin per pair), which
// the rotated dims then replace; threads 0..31, each reading its own pair.
__device__ __forceinline__ void block_rope_inplace(const float *row, float *rot) {
  const int t = threadIdx.x;
  if (t < 32) {
    float a = row[kLat + 2 * t], bb = row[kLat + 2 * t + 1];
    rope_pair(a, bb, rot[2 * t], rot[2 * t + 1]);
    rot[2 * t] = a;
    rot[2 * t + 1] = bb;
  }
}

// Two values of an NVFP4 group of 16 held by 8 consecutive lanes: returns the
// packed byte (first value in the low nibble); *sc = the group's scale code.
__device__ __forceinline__ uint32_t nvfp4_pair(float x0, float x1, uint32_t *sc) {
  float amax = fmaxf(fabsf(x0), fabsf(x1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  uint32_t code = e4m3_code(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_value(code);
  if (s == 0.0f) {
    *sc = 0;
    return 0;
  }
  *sc = code;
  return e2m1_code(__fdiv_rn(x0, s)) | (e2m1_code(__fdiv_rn(x1, s)) << 4);
}

// Entry e of sequence b from row[0:704] (smem: main vector, RoPE dims
// unrotated, then the indexer key) and rot[0:64] (smem, rotated RoPE dims).
__device__ __forceinline__ void block_encode_entry(const csa2_cache &c, int b, int64_t e, const float *row,
                                                   const float *rot, int32_t *err) {
  const int t = threadIdx.x, lane = t & 31;
  const EntryMap map = entry_map(c);
  const int64_t pe = phys_entry(map, b, e), pt = phys_tile(map, b, e / kIdxTile);
  if (pe < 0 || pt < 0) {  // a page id outside the pool: nothing written
    if (t == 0) raise_err(err, CSA2_DEVERR_INDEX);
    return;
  }
  const size_t ent = static_cast<size_t>(pe);
  uint32_t sc;
  if (c.entry_format == CSA2_ENTRY_FP8) {
    // V4 entry: latent MXFP8 block g (32 dims) on warp g % 8, one dim per lane
    const int warp = t >> 5;
    for (int g = warp; g < 16; g += kEncThreads / 32) {
      const float x = row[32 * g + lane];
      float amax = fabsf(x);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      uint32_t code = 0;
      sc = 0;
      if (amax != 0.0f) {
        int ex = floor_log2f(amax) - 8;
        ex = max(-127, min(127, ex));
        code = e4m3_code(__fmul_rn(x, pow2f(-ex)));
        sc = static_cast<uint32_t>(ex + 127);
      }
      uint32_t w = code << (8 * (lane & 3));  // four lanes' bytes into one word
      w |= __shfl_xor_sync(0xffffffffu, w, 1);
      w |= __shfl_xor_sync(0xffffffffu, w, 2);
      if ((lane & 3) == 0) reinterpret_cast<uint32_t *>(c.lat_codes + ent * 512 + 32 * g)[lane >> 2] = w;
      if (lane == 0) c.lat_scales[ent * 16 + g] = static_cast<uint8_t>(sc);
    }
    if (t < 64) reinterpret_cast<__nv_bfloat16 *>(c.rope_codes + ent * 128)[t] = __float2bfloat16_rn(rot[t]);
  } else {
    {  // latent: thread t has dims 2t, 2t+1 (group t / 8)
      const float2 v = reinterpret_cast<const float2 *>(row)[t];
      const uint32_t byte = nvfp4_pair(v.x, v.y, &sc);
      c.lat_codes[ent * 256 + t] = static_cast<uint8_t>(byte);
      if ((t & 7) == 0) c.lat_scales[ent * 32 + (t >> 3)] = static_cast<uint8_t>(sc);
    }
    if (t < 32) {  // RoPE sidecar: rotated dims 2t, 2t+1 (group t / 8)
      const float2 v = reinterpret_cast<const float2 *>(rot)[t];
      const uint32_t byte = nvfp4_pair(v.x, v.y, &sc);
      c.rope_codes[ent * 32 + t] = static_cast<uint8_t>(byte);
      if ((t & 7) == 0) c.rope_scales[ent * 4 + (t >> 3)] = static_cast<uint8_t>(sc);
    }
  }
  if (t >= 32 && t < 64) {  // indexer key, MXFP4: lane l has dims 4l..4l+3 (block l / 8)
    const float4 v = reinterpret_cast<const float4 *>(row + kDqk)[lane];
    const float x[4] = {v.x, v.y, v.z, v.w};
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    uint32_t codes = 0;
    sc = 0;
    if (amax != 0.0f) {
      int ex = floor_log2f(amax) - 2;
      ex = max(-127, min(127, ex));
      const float inv = pow2f(-ex);
#pragma unroll
      for (int i = 0; i < 4; ++i) codes |= e2m1_code(__fmul_rn(x[i], inv)) << (4 * i);
      sc = static_cast<uint32_t>(ex + 127);
    }
    const int blk = lane >> 3;
    *reinterpret_cast<uint16_t *>(c.idx_codes + idx_code_at(pt, e % kIdxTile, blk) + 2 * (lane & 7)) =
        static_cast<uint16_t>(codes);
    if ((lane & 7) == 0) c.idx_scales[idx_scale_at(pt, e % kIdxTile) + blk] = static_cast<uint8_t>(sc);
  }
}

// One window token from row[0:512] (smem) and rot[0:64] (smem) into codes
// (576 B MXFP8 or 1152 B bf16) and scales (18 B, MXFP8).
__device__ __forceinline__ void block_encode_swa(uint8_t *codes, uint8_t *scales, int swa_dtype, const float *row,
                                                 const float *rot) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (swa_dtype == CSA2_SWA_MXFP8) {
    // group g (32 dims) on warp g % 8, one dim per lane
    for (int g = warp; g < 18; g += kEncThreads / 32) {
      const int d = 32 * g + lane;
      const float x = d < kLat ? row[d] : rot[d - kLat];
      float amax = fabsf(x);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      uint32_t code = 0, sc = 0;
      if (amax != 0.0f) {
        int ex = floor_log2f(amax) - 8;
        ex = max(-127, min(127, ex));
        code = e4m3_code(__fmul_rn(x, pow2f(-ex)));
        sc = static_cast<uint32_t>(ex + 127);
      }
      // four lanes' bytes into one word
      uint32_t w = code << (8 * (lane & 3));
      w |= __shfl_xor_sync(0xffffffffu, w, 1);
      w |= __shfl_xor_sync(0xffffffffu, w, 2);
      if ((lane & 3) == 0) reinterpret_cast<uint32_t *>(codes + 32 * g)[lane >> 2] = w;
      if (lane == 0) scales[g] = static_cast<uint8_t>(sc);
    }
  } else {
    __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(codes);
    for (int d = t; d < kDqk; d += kEncThreads) h[d] = __float2bfloat16_rn(d < kLat ? row[d] : rot[d - kLat]);
  }
}

}  // namespace csa2
