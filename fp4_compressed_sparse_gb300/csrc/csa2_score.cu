// csa2_score.cu -- lightning-indexer scores, FULL and POOL modes.
//
// [P5] "DeepSeek-V4: Towards Highly Efficient Million-Token Context
// Intelligence" §2.3.1 "Sparse Selection을 위한 Lightning Indexer":
//   I_{t,s} = sum_h w_{t,h} * ReLU(q_{t,h} . K_s),  visible iff s < floor(t/m);
// §2.3.4: the indexer QK product runs in FP4, so q is quantised to MXFP4 like K.
// [P1] "DeepSeek V4.1 Flash 아키텍처 분석" §"512개를 고르기 위해 ..." (POOL:
// Reindex layers score only the 2,048 x 8 candidate positions).
//
// CUDA-core path: every (query head, key) dot is an exact integer sum of
// products of doubled E2M1 codes (dp4a), per 32-wide block, scaled by
// 2^(eq+ek-2).  The four block terms and the fp32 sum are exact whenever the
// block exponents of the pair span <= 9 binades, so d_h equals the fp32 value of
// the exact dot; a visible key whose pair with some head exceeds that span
// raises CSA2_DEVERR_INEXACT (blocks with scale code 0 take no part, as in the
// tensor-core path).  The head reduction is the fixed-order chain
// acc = fma(w_h, max(d_h, +0), acc).
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 128;  // one key per thread
constexpr int kMaxExactSpan = 9;

// max - min of the nonzero E8M0 codes packed in w (0 if fewer than two)
__device__ __forceinline__ int span4(uint32_t w) {
  int mx = 0, mn = 255;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = static_cast<int>((w >> (8 * j)) & 0xFFu);
    if (c) {
      mx = max(mx, c);
      mn = min(mn, c);
    }
  }
  return mx >= mn ? mx - mn : 0;
}
// span of e_q,j + e_k,j over the blocks where both codes are nonzero
__device__ __forceinline__ int pair_span4(uint32_t wq, uint32_t wk) {
  int mx = 0, mn = 1024;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int cq = static_cast<int>((wq >> (8 * j)) & 0xFFu), ck = static_cast<int>((wk >> (8 * j)) & 0xFFu);
    if (cq && ck) {
      mx = max(mx, cq + ck);
      mn = min(mn, cq + ck);
    }
  }
  return mx >= mn ? mx - mn : 0;
}

__global__ void __launch_bounds__(kThreads) k_index_score_dp4a(ScoreArgs a) {
  extern __shared__ uint32_t smem[];
  const int H = a.heads;
  uint32_t *s_q = smem;                                          // [H][32] int8x4 words (2*E2M1 of q)
  float *s_qf = reinterpret_cast<float *>(s_q + H * 32);          // [H][4] 2^(eq-1)
  float *s_w = s_qf + H * 4;                                      // [H]
  uint32_t *s_qc = reinterpret_cast<uint32_t *>(s_w + H);         // [H] the four block scale codes

  const int r = blockIdx.y;
  const int64_t T = a.q_pos[r] / a.ratio;  // visible entries
  const int64_t slot0 = static_cast<int64_t>(blockIdx.x) * kThreads;
  const bool pool_mode = a.pool != nullptr;
  if (!pool_mode && T > a.cap && blockIdx.x == 0 && threadIdx.x == 0) raise_err(a.err, CSA2_DEVERR_INDEX);
  const int64_t nslots = pool_mode ? static_cast<int64_t>(a.pool_blocks) * a.pool_bs : min(T, min(a.cap, a.stride));
  if (slot0 >= nslots) return;
  const int seq = a.cache_seq < 0 ? r : a.cache_seq;

  // quantise this row's indexer query: H heads x 4 MXFP4 blocks
  for (int task = threadIdx.x; task < H * 4; task += kThreads) {
    const int h = task >> 2, blk = task & 3;
    const uint16_t *src = a.q_idx + (static_cast<size_t>(r) * H + h) * kDi + 32 * blk;
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(static_cast<uint32_t>(src[i]) << 16);
    uint32_t w4[4], sc;
    quant_mxfp4_32(x, w4, &sc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s_q[h * 32 + blk * 8 + 2 * i] = e2m1x4_twice_i8(w4[i] & 0xFFFFu);
      s_q[h * 32 + blk * 8 + 2 * i + 1] = e2m1x4_twice_i8(w4[i] >> 16);
    }
    s_qf[h * 4 + blk] = pow2f(static_cast<int>(sc) - 128);
    reinterpret_cast<uint8_t *>(s_qc + h)[blk] = static_cast<uint8_t>(sc);
  }
  for (int h = threadIdx.x; h < H; h += kThreads) s_w[h] = a.w[static_cast<size_t>(r) * H + h];
  __syncthreads();

  const int64_t slot = slot0 + threadIdx.x;
  if (slot >= nslots) return;
  int64_t s = slot;
  if (pool_mode) {
    const int32_t pid = a.pool[static_cast<size_t>(r) * a.pool_blocks + slot / a.pool_bs];
    if (pid < 0) return;
    s = static_cast<int64_t>(pid) * a.pool_bs + slot % a.pool_bs;
    if (s >= a.cap) {
      raise_err(a.err, CSA2_DEVERR_INDEX);
      return;
    }
    if (s >= T) return;
  }
  const int64_t pt = phys_tile(a.map, seq, s / kIdxTile);
  if (pt < 0) {  // a page id outside the pool
    raise_err(a.err, CSA2_DEVERR_INDEX);
    return;
  }
  const int mrow = static_cast<int>(s % kIdxTile);
  const uint32_t ksc = *reinterpret_cast<const uint32_t *>(a.idx_scales + idx_scale_at(pt, mrow));
  uint32_t kw[32];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 u = *reinterpret_cast<const uint4 *>(a.idx_codes + idx_code_at(pt, mrow, v));
    const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kw[8 * v + 2 * i] = e2m1x4_twice_i8(words[i] & 0xFFFFu);
      kw[8 * v + 2 * i + 1] = e2m1x4_twice_i8(words[i] >> 16);
    }
  }
  float kf[4];
#pragma unroll
  for (int blk = 0; blk < 4; ++blk) kf[blk] = pow2f(static_cast<int>((ksc >> (8 * blk)) & 0xFFu) - 128);

  // exactness bound: the sum of the query's and the key's spans bounds every
  // pair's; only when it fails is each head checked
  {
    int qmax = 0;
    for (int h = 0; h < H; ++h) qmax = max(qmax, span4(s_qc[h]));
    if (qmax + span4(ksc) > kMaxExactSpan) {
      bool bad = false;
      for (int h = 0; h < H && !bad; ++h) bad = pair_span4(s_qc[h], ksc) > kMaxExactSpan;
      if (bad) raise_err(a.err, CSA2_DEVERR_INEXACT);
    }
  }

  float acc = 0.0f;
  for (int h = 0; h < H; ++h) {
    float t[4];
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      int isum = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w)
        isum = __dp4a(static_cast<int>(kw[8 * blk + w]), static_cast<int>(s_q[h * 32 + 8 * blk + w]), isum);
      t[blk] = __fmul_rn(__fmul_rn(__int2float_rn(isum), s_qf[h * 4 + blk]), kf[blk]);
    }
    const float d = __fadd_rn(__fadd_rn(__fadd_rn(t[0], t[1]), t[2]), t[3]);
    const float rl = d > 0.0f ? d : 0.0f;
    acc = __fmaf_rn(s_w[h], rl, acc);
  }
  a.scores[static_cast<size_t>(r) * a.stride + slot] = acc;
}

}  // namespace

cudaError_t launch_index_score(const ScoreArgs &a, cudaStream_t s) {
  const int64_t nslots = a.pool ? static_cast<int64_t>(a.pool_blocks) * a.pool_bs : a.stride;
  if (nslots <= 0 || a.rows <= 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>((nslots + kThreads - 1) / kThreads), a.rows);
  const size_t smem = static_cast<size_t>(a.heads) * (32 * 4 + 4 * 4 + 4 + 4);
  k_index_score_dp4a<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace csa2
