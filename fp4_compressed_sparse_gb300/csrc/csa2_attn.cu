// csa2_attn.cu -- sparse absorbed-query attention over the selected FP4 entries
// plus the sliding window, with an optional attention sink.
//
// [P5] "DeepSeek-V4: Towards Highly Efficient Million-Token Context
// Intelligence" §2.3.1 "Shared Key-Value MQA" (each selected entry is key and
// value), §2.3.3 (window branch; sink exp(z'_h) in the denominator);
// [P2] "DeepSeek Multi-Head Latent Attention(MLA) 해부" §4 (absorbed query: the
// logit is q_lat . c + q_rope . k_rope, the value is the 512-dim latent c).
//
// One CTA = (16 heads, one split of the entry list, one row).  Entries are
// gathered 32 at a time and dequantised exactly into shared memory (bf16 for
// the 576-dim keys, fp16 for the 512-dim values: an E2M1 code times an E4M3 or
// E8M0 scale has at most 6 significant bits), then
//   S = Q K^T   (mma.sync m16n8k16 bf16, fp32 accumulate; warp w owns 8 entries)
//   online softmax in the log2 domain (fp32)
//   O += P V    (mma.sync m16n8k16 fp16, fp32 accumulate; warp w owns 128 dims)
// Splits write unnormalised partials (O, m, l) and a combine kernel merges them
// (flash-decoding LSE merge) and applies the sink.
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 128;
constexpr int kEnt = 32;         // entries per chunk
constexpr int kQS = kDqk + 8;    // bf16 row stride (odd multiple of 16 B: conflict-free ldmatrix)
constexpr int kVS = kLat + 8;    // fp16 row stride
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Smem {
  __nv_bfloat16 q[16][kQS];
  __nv_bfloat16 k[kEnt][kQS];
  __half v[kEnt][kVS];
  float s[16][kEnt + 1];
  int64_t src[kEnt];
  int kind[kEnt];  // 0 empty, 1 cache entry, 2 window ring slot, 3 window linear row
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void put(Smem &sm, int e, int d, float v) {
  sm.k[e][d] = __float2bfloat16_rn(v);
  if (d < kLat) sm.v[e][d] = __float2half_rn(v);
}

// Dequantise entry e (kind/src resolved) into sm.k / sm.v; `part` in 0..3.
__device__ __forceinline__ void load_entry(const AttnArgs &a, Smem &sm, int e, int part) {
  const int kind = sm.kind[e];
  const int64_t src = sm.src[e];
  if (kind == 1) {
    const uint4 *cp = reinterpret_cast<const uint4 *>(a.lat_codes + src * 256 + part * 64);
    const uint2 sc8 = *reinterpret_cast<const uint2 *>(a.lat_scales + src * 32 + part * 8);
    const uint32_t scw[2] = {sc8.x, sc8.y};
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 u = cp[v];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // word q of uint4 v holds dims part*128 + 32v + 8q .. +7 (group 2v + q/2)
        const int g = 2 * v + (q >> 1);
        const float s = e4m3_value((scw[g >> 2] >> (8 * (g & 3))) & 0xFFu);
        const int d0 = part * 128 + 32 * v + 8 * q;
#pragma unroll
        for (int i = 0; i < 8; ++i) put(sm, e, d0 + i, e2m1_value((w[q] >> (4 * i)) & 15u) * s);
      }
    }
    const uint2 rc = *reinterpret_cast<const uint2 *>(a.rope_codes + src * 32 + part * 8);
    const float rs = e4m3_value(a.rope_scales[src * 4 + part]);
    const uint32_t rw[2] = {rc.x, rc.y};
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i) put(sm, e, kLat + 16 * part + 8 * q + i, e2m1_value((rw[q] >> (4 * i)) & 15u) * rs);
  } else if (kind == 2 || kind == 3) {
    const uint8_t *codes;
    const uint8_t *scales;
    if (kind == 2) {
      codes = a.ring_codes + src * (a.swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152);
      scales = a.ring_scales ? a.ring_scales + src * kSwaScaleStride : nullptr;
    } else {
      codes = a.lin_codes + src * (a.swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152);
      scales = a.lin_scales ? a.lin_scales + src * kSwaScaleStride : nullptr;
    }
    const int d0 = part * 144;
    if (a.swa_dtype == CSA2_SWA_MXFP8) {
      const uint4 *cp = reinterpret_cast<const uint4 *>(codes + d0);
#pragma unroll
      for (int v = 0; v < 9; ++v) {
        const uint4 u = cp[v];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int d = d0 + 16 * v + 4 * q + i;
            put(sm, e, d, e4m3_value((w[q] >> (8 * i)) & 0xFFu) * e8m0_value(scales[d >> 5]));
          }
      }
    } else {
      const uint4 *cp = reinterpret_cast<const uint4 *>(codes + 2 * d0);
#pragma unroll
      for (int v = 0; v < 18; ++v) {
        const uint4 u = cp[v];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int d = d0 + 8 * v + 2 * q;
          put(sm, e, d, __uint_as_float(w[q] << 16));
          put(sm, e, d + 1, __uint_as_float(w[q] & 0xFFFF0000u));
        }
      }
    }
  } else {
    for (int d = part * 144; d < part * 144 + 144; ++d) put(sm, e, d, 0.0f);
  }
}

__global__ void __launch_bounds__(kThreads) k_attn(AttnArgs a, int n_splits, int per_split) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int hg = blockIdx.x, split = blockIdx.y, row = blockIdx.z;
  const int H = a.heads;
  const int seq = a.cache_seq < 0 ? row : a.cache_seq;
  const int64_t qpos = a.q_pos[row];
  const int64_t T = qpos / a.ratio;
  const int64_t ntok = a.n_tokens[seq];
  const int64_t lin_base = a.lin_base ? *a.lin_base : INT64_MAX;
  const int L = a.k + kWin;
  const int e_begin = split * per_split;
  const int e_end = min(L, e_begin + per_split);
  const float scale2 = a.sm_scale * kLog2e;

  // Q rows of this head group
  {
    const uint4 *qsrc = reinterpret_cast<const uint4 *>(a.q + (static_cast<size_t>(row) * H + hg * 16) * kDqk);
    for (int i = tid; i < 16 * 72; i += kThreads) {
      const int r = i / 72, c = i % 72;
      *reinterpret_cast<uint4 *>(&sm.q[r][8 * c]) = qsrc[r * 72 + c];
    }
  }

  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};

  for (int c0 = e_begin; c0 < e_end; c0 += kEnt) {
    __syncthreads();  // previous chunk fully consumed (and Q stored on the first pass)
    if (tid < kEnt) {
      const int j = c0 + tid;
      int kind = 0;
      int64_t src = 0;
      if (j < e_end) {
        if (j < a.k) {
          const int32_t s = a.idx[static_cast<size_t>(row) * a.k + j];
          if (s >= 0) {
            if (s < T && s < a.cap) {
              kind = 1;
              src = static_cast<int64_t>(seq) * a.cap + s;
            } else {
              raise_err(a.err, CSA2_DEVERR_INDEX);
            }
          }
        } else {
          const int64_t tok = qpos - (kWin - 1) + (j - a.k);
          if (tok >= 0 && tok < ntok && tok <= qpos) {
            if (tok >= lin_base) {
              kind = 3;
              src = tok - lin_base;
            } else {
              kind = 2;
              src = static_cast<int64_t>(a.ring_single ? 0 : seq) * kWin + (tok % kWin);
            }
          }
        }
      }
      sm.kind[tid] = kind;
      sm.src[tid] = src;
    }
    __syncthreads();
    load_entry(a, sm, tid >> 2, tid & 3);
    __syncthreads();

    // S = Q K^T for entries 8*warp .. 8*warp+7
    {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t qa = smem_u32(&sm.q[lane & 15][(lane >> 4) * 8]);
      const uint32_t kb = smem_u32(&sm.k[8 * warp + (lane & 7)][((lane >> 3) & 1) * 8]);
#pragma unroll 4
      for (int kk = 0; kk < kDqk / 16; ++kk) {
        uint32_t a0, a1, a2, a3, b0, b1;
        ldsm_x4(qa + kk * 32, a0, a1, a2, a3);
        ldsm_x2(kb + kk * 32, b0, b1);
        mma_bf16(acc, a0, a1, a2, a3, b0, b1);
      }
      sm.s[g][8 * warp + 2 * t] = acc[0] * scale2;
      sm.s[g][8 * warp + 2 * t + 1] = acc[1] * scale2;
      sm.s[g + 8][8 * warp + 2 * t] = acc[2] * scale2;
      sm.s[g + 8][8 * warp + 2 * t + 1] = acc[3] * scale2;
    }
    __syncthreads();

    // online softmax (every warp redundantly for its two rows g, g+8)
    float p[2][2][4];  // [row g/g+8][kk][4 cols]
    float rmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int col = kk * 16 + 2 * t + (c & 1) + (c >> 1) * 8;
        const bool ok = sm.kind[col] != 0;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const float v = ok ? sm.s[g + 8 * rr][col] : -INFINITY;
          p[rr][kk][c] = v;
          rmax[rr] = fmaxf(rmax[rr], v);
        }
      }
    float alpha[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      rmax[rr] = fmaxf(rmax[rr], __shfl_xor_sync(0xffffffffu, rmax[rr], 1));
      rmax[rr] = fmaxf(rmax[rr], __shfl_xor_sync(0xffffffffu, rmax[rr], 2));
      const float m_new = fmaxf(m_run[rr], rmax[rr]);
      alpha[rr] = (m_new == -INFINITY) ? 1.0f : exp2f(m_run[rr] - m_new);
      float sum = 0.0f;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float e = (m_new == -INFINITY) ? 0.0f : exp2f(p[rr][kk][c] - m_new);
          p[rr][kk][c] = e;
          sum += e;
        }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      l_run[rr] = l_run[rr] * alpha[rr] + sum;
      m_run[rr] = m_new;
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }

    // O += P V for dims 128*warp .. +127
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t a0 = pack_half2(p[0][kk][0], p[0][kk][1]);
      const uint32_t a1 = pack_half2(p[1][kk][0], p[1][kk][1]);
      const uint32_t a2 = pack_half2(p[0][kk][2], p[0][kk][3]);
      const uint32_t a3 = pack_half2(p[1][kk][2], p[1][kk][3]);
      const uint32_t vb =
          smem_u32(&sm.v[kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8][128 * warp + (lane >> 4) * 8]);
#pragma unroll
      for (int n = 0; n < 16; n += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + n * 16, b0, b1, b2, b3);
        mma_f16(o[n], a0, a1, a2, a3, b0, b1);
        mma_f16(o[n + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }

  // epilogue
  const int h0 = hg * 16 + g, h1 = h0 + 8;
  if (n_splits == 1) {
    float inv[2], lse_v[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int h = rr ? h1 : h0;
      float m = m_run[rr], l = l_run[rr], f = 1.0f;
      if (a.sink) {
        const float s2 = a.sink[h] * kLog2e;
        const float mf = fmaxf(m, s2);
        f = (m == -INFINITY) ? 0.0f : exp2f(m - mf);
        l = l * f + exp2f(s2 - mf);
        m = mf;
      }
      inv[rr] = l > 0.0f ? f / l : 0.0f;
      lse_v[rr] = l > 0.0f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
    float *out0 = a.out + (static_cast<size_t>(row) * H + h0) * kLat;
    float *out1 = a.out + (static_cast<size_t>(row) * H + h1) * kLat;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int d = 128 * warp + 8 * n + 2 * t;
      *reinterpret_cast<float2 *>(out0 + d) = make_float2(o[n][0] * inv[0], o[n][1] * inv[0]);
      *reinterpret_cast<float2 *>(out1 + d) = make_float2(o[n][2] * inv[1], o[n][3] * inv[1]);
    }
    if (warp == 0 && t == 0) {
      a.lse[static_cast<size_t>(row) * H + h0] = lse_v[0];
      a.lse[static_cast<size_t>(row) * H + h1] = lse_v[1];
    }
  } else {
    const size_t base = (static_cast<size_t>(row) * n_splits + split) * H;
    float *po = a.part;                                                       // [rows][splits][H][512]
    float *pml = a.part + static_cast<size_t>(a.rows) * n_splits * H * kLat;  // [rows][splits][H][2]
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int d = 128 * warp + 8 * n + 2 * t;
      *reinterpret_cast<float2 *>(po + (base + h0) * kLat + d) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2 *>(po + (base + h1) * kLat + d) = make_float2(o[n][2], o[n][3]);
    }
    if (warp == 0 && t == 0) {
      *reinterpret_cast<float2 *>(pml + (base + h0) * 2) = make_float2(m_run[0], l_run[0]);
      *reinterpret_cast<float2 *>(pml + (base + h1) * 2) = make_float2(m_run[1], l_run[1]);
    }
  }
}

// LSE merge of the split partials: grid (H, rows), 128 threads x 4 dims.
__global__ void __launch_bounds__(128) k_attn_combine(AttnArgs a, int n_splits) {
  const int h = blockIdx.x, row = blockIdx.y, H = a.heads;
  const float *po = a.part;
  const float *pml = a.part + static_cast<size_t>(a.rows) * n_splits * H * kLat;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, pml[((static_cast<size_t>(row) * n_splits + s) * H + h) * 2]);
  const float s2 = a.sink ? a.sink[h] * kLog2e : -INFINITY;
  M = fmaxf(M, s2);
  float L = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const size_t base = (static_cast<size_t>(row) * n_splits + s) * H + h;
      const float m = pml[base * 2], l = pml[base * 2 + 1];
      if (m == -INFINITY) continue;
      const float f = exp2f(m - M);
      L += l * f;
      const float4 v = reinterpret_cast<const float4 *>(po + base * kLat)[threadIdx.x];
      acc.x += v.x * f;
      acc.y += v.y * f;
      acc.z += v.z * f;
      acc.w += v.w * f;
    }
    if (a.sink) L += exp2f(s2 - M);
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  reinterpret_cast<float4 *>(a.out + (static_cast<size_t>(row) * H + h) * kLat)[threadIdx.x] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (threadIdx.x == 0) a.lse[static_cast<size_t>(row) * H + h] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

int choose_splits(int rows, int heads, int k) {
  const int L = k + kWin;
  const int ctas = rows * (heads / 16);
  if (ctas >= 120) return 1;            // the rows alone fill most of the 152 SMs
  int s = (2 * 152 + ctas - 1) / ctas;  // aim for ~2 CTAs per SM
  const int max_s = (L + 63) / 64;      // at least 64 entries per split
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  return s;
}

}  // namespace

size_t attn_workspace_bytes(int rows, int heads, int k) {
  const int s = choose_splits(rows, heads, k);
  if (s == 1) return 256;
  return static_cast<size_t>(rows) * s * heads * (kLat + 2) * sizeof(float) + 256;
}

cudaError_t launch_attn(const AttnArgs &a0, void *ws, size_t ws_bytes, cudaStream_t st) {
  if (a0.rows <= 0) return cudaSuccess;
  AttnArgs a = a0;
  const int n_splits = choose_splits(a.rows, a.heads, a.k);
  const int L = a.k + kWin;
  int per = (L + n_splits - 1) / n_splits;
  per = (per + kEnt - 1) / kEnt * kEnt;
  a.part = static_cast<float *>(ws);
  static bool attr_set = false;
  const int smem = static_cast<int>(sizeof(Smem));
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_attn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(a.heads / 16, n_splits, a.rows);
  k_attn<<<grid, kThreads, smem, st>>>(a, n_splits, per);
  if (n_splits > 1) k_attn_combine<<<dim3(a.heads, a.rows), 128, 0, st>>>(a, n_splits);
  (void)ws_bytes;
  return cudaGetLastError();
}

}  // namespace csa2
