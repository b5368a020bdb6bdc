// csa2_append.cu -- csa2_kv_append kernels: RoPE, then quantise new tokens into
// the FP4 cache (288 B main entry + 36 B RoPE sidecar + 68 B MXFP4 indexer key)
// and the 8-bit / bf16 sliding-window ring.
//
// [P1] "DeepSeek V4.1 Flash 아키텍처 분석" §"890 bytes/token은 어떻게 나오는가"
//      (record formats); [P4] "매개변수는 커졌는데 메모리는 4분의 1 ..."
//      §"890이 맞아떨어지는 계산" (quantise after RoPE); [P5] "DeepSeek-V4 ..."
//      §2.3.1 (overlapping compression, m = 2) and §3.5.1 (compression buffer,
//      fixed-size window state).
//
// Ratio 1: one 256-thread block encodes one token (entry and window slot), each
// thread a few values.  Ratio 2: one warp encodes one compressed entry (or one
// window token): lane l quantises latent group l (16 values), lanes 0..3 the
// four RoPE groups, lanes 4..7 the four MXFP4 indexer blocks.
#include "csa2_encode.cuh"
#include "csa2_internal.cuh"

namespace csa2 {

namespace {

constexpr int kWarps = 8;  // tokens per 256-thread block

__device__ __forceinline__ float load_in(const void *p, size_t i, int in_bf16) {
  if (in_bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
  return reinterpret_cast<const float *>(p)[i];
}

// Whether sequence b may take n_new more tokens (capacity in entries, RoPE table).
__device__ __forceinline__ bool append_ok(const csa2_cache &c, int64_t t0, int n_new, int64_t rope_len) {
  return (t0 + n_new) / c.ratio <= static_cast<int64_t>(c.capacity) && t0 + n_new <= rope_len;
}

__device__ __forceinline__ void append_fail(const csa2_cache &c, int64_t t0, int n_new, int64_t rope_len,
                                            int32_t *err) {
  if ((t0 + n_new) / c.ratio > static_cast<int64_t>(c.capacity)) raise_err(err, CSA2_DEVERR_CAPACITY);
  else raise_err(err, CSA2_DEVERR_ROPE);
}

}  // namespace

namespace {

// Ratio 1: token t is entry t.  grid (n_new, batch), one 256-thread block per
// token.  `advance`: this launch is the only one of the append (one token per
// sequence), so the block also moves n_tokens on once it is done.
__global__ void __launch_bounds__(kEncThreads) k_append_r1(csa2_cache c, const void *kv, const void *ik, int in_bf16,
                                                           const float *rope_cs, int64_t rope_len, int n_new,
                                                           int advance, int32_t *err) {
  __shared__ __align__(16) float row[kDcmp];
  __shared__ __align__(16) float rot[kRope];
  const int b = blockIdx.y, j = blockIdx.x;
  // the token's rows do not depend on the token count: request them together
  // with it, so that the RoPE row (which does) is the only later round trip
  const int64_t t0 = c.n_tokens[b];
  const size_t base = static_cast<size_t>(b) * n_new + j;
  for (int i = threadIdx.x; i < kDqk; i += blockDim.x) row[i] = load_in(kv, base * kDqk + i, in_bf16);
  for (int i = threadIdx.x; i < kDi; i += blockDim.x) row[kDqk + i] = load_in(ik, base * kDi + i, in_bf16);
  const bool ok = append_ok(c, t0, n_new, rope_len);
  const int64_t t = t0 + j;
  float cs = 0.0f;  // this thread's RoPE table value (threads 0..63)
  if (ok && threadIdx.x < 64) cs = rope_cs[t * 64 + threadIdx.x];
  if (!ok) {
    if (j == 0 && threadIdx.x == 0) append_fail(c, t0, n_new, rope_len, err);
    return;
  }
  if (threadIdx.x < 64) rot[threadIdx.x] = cs;  // staged through rot, rotated in place below
  __syncthreads();
  block_rope_inplace(row, rot);
  __syncthreads();
  block_encode_entry(c, b, t, row, rot, err);
  if (j >= n_new - kWin) {
    const size_t slot = static_cast<size_t>(b) * kWin + (t % kWin);
    block_encode_swa(c.swa_codes + slot * (c.swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152),
                     c.swa_scales ? c.swa_scales + slot * kSwaScaleStride : nullptr, c.swa_dtype, row, rot);
  }
  if (advance) {
    __syncthreads();  // every thread has read n_tokens
    if (threadIdx.x == 0) c.n_tokens[b] = t0 + n_new;
  }
}

// Compression row `which` (0 C^a, 1 C^b, 2 Z^a, 3 Z^b) of token p: from this
// call's input when p >= t0, else from the compression buffer (slot p % 4).
__device__ __forceinline__ const float *cmp_row(const csa2_cache &c, const csa2_compress_in &in, int b,
                                                int n_new, int64_t t0, int64_t p, int which) {
  if (p >= t0) {
    const float *src = which == 0 ? in.ca : which == 1 ? in.cb : which == 2 ? in.za : in.zb;
    return src + (static_cast<size_t>(b) * n_new + (p - t0)) * kDcmp;
  }
  return c.cmp_buf + ((static_cast<size_t>(b) * 4 + (p & 3)) * 4 + which) * kDcmp;
}

// Ratio 2: entry i from tokens 2i, 2i+1 (a rows) and 2i-2, 2i-1 (b rows).
// grid (ceil((n_new/2+1)/8), batch), 256 threads.
__global__ void __launch_bounds__(256) k_append_r2_entries(csa2_cache c, csa2_compress_in in, const float *rope_cs,
                                                           int64_t rope_len, int n_new, float *dbg,
                                                           int32_t *err) {
  __shared__ float srow[kWarps][kDcmp];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int e = blockIdx.x * kWarps + warp;
  const int64_t t0 = c.n_tokens[b];
  if (!append_ok(c, t0, n_new, rope_len)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) append_fail(c, t0, n_new, rope_len, err);
    return;
  }
  const int64_t i0 = t0 / 2;
  const int64_t n_emit = (t0 + n_new) / 2 - i0;
  if (e >= n_emit) return;
  const int64_t i = i0 + e;
  const float *a0c = cmp_row(c, in, b, n_new, t0, 2 * i, 0), *a1c = cmp_row(c, in, b, n_new, t0, 2 * i + 1, 0);
  const float *a0z = cmp_row(c, in, b, n_new, t0, 2 * i, 2), *a1z = cmp_row(c, in, b, n_new, t0, 2 * i + 1, 2);
  const bool has_b = i > 0;
  const float *b0c = has_b ? cmp_row(c, in, b, n_new, t0, 2 * i - 2, 1) : nullptr;
  const float *b1c = has_b ? cmp_row(c, in, b, n_new, t0, 2 * i - 1, 1) : nullptr;
  const float *b0z = has_b ? cmp_row(c, in, b, n_new, t0, 2 * i - 2, 3) : nullptr;
  const float *b1z = has_b ? cmp_row(c, in, b, n_new, t0, 2 * i - 1, 3) : nullptr;
  float *dst_dbg = dbg ? dbg + (static_cast<size_t>(b) * (n_new / 2 + 1) + e) * kDcmp : nullptr;
  for (int j = lane; j < kDcmp; j += 32) {
    // per-channel softmax over the 4 rows, in fp64, rounded once to fp32
    double l0 = __dadd_rn(static_cast<double>(a0z[j]), static_cast<double>(in.ba[j]));
    double l1 = __dadd_rn(static_cast<double>(a1z[j]), static_cast<double>(in.ba[kDcmp + j]));
    double l2 = has_b ? __dadd_rn(static_cast<double>(b0z[j]), static_cast<double>(in.bb[j])) : -INFINITY;
    double l3 = has_b ? __dadd_rn(static_cast<double>(b1z[j]), static_cast<double>(in.bb[kDcmp + j])) : -INFINITY;
    double mx = fmax(fmax(l0, l1), fmax(l2, l3));
    double e0 = exp(__dadd_rn(l0, -mx)), e1 = exp(__dadd_rn(l1, -mx));
    double e2 = has_b ? exp(__dadd_rn(l2, -mx)) : 0.0, e3 = has_b ? exp(__dadd_rn(l3, -mx)) : 0.0;
    double den = __dadd_rn(__dadd_rn(__dadd_rn(__dadd_rn(0.0, e0), e1), e2), e3);
    double acc = 0.0;
    acc = __dadd_rn(acc, __dmul_rn(__ddiv_rn(e0, den), static_cast<double>(a0c[j])));
    acc = __dadd_rn(acc, __dmul_rn(__ddiv_rn(e1, den), static_cast<double>(a1c[j])));
    acc = __dadd_rn(acc, __dmul_rn(__ddiv_rn(e2, den), has_b ? static_cast<double>(b0c[j]) : 0.0));
    acc = __dadd_rn(acc, __dmul_rn(__ddiv_rn(e3, den), has_b ? static_cast<double>(b1c[j]) : 0.0));
    const float v = __double2float_rn(acc);
    srow[warp][j] = v;
    if (dst_dbg) dst_dbg[j] = v;
  }
  __syncwarp();
  warp_encode_entry(c, b, i, srow[warp], rope_cs + (2 * i) * 64, lane, err);
}

// Ratio 2 tail: window slots of the last min(n_new,128) tokens (their own C^a
// rows, rotated at t) and the compression buffer rows of the last 4 tokens.
__global__ void __launch_bounds__(256) k_append_r2_tail(csa2_cache c, csa2_compress_in in, const float *rope_cs,
                                                        int64_t rope_len, int n_new) {
  __shared__ float srow[kWarps][kDqk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int64_t t0 = c.n_tokens[b];
  if (!append_ok(c, t0, n_new, rope_len)) return;
  const int n_tail = min(n_new, kWin);
  const int idx = blockIdx.x * kWarps + warp;
  if (idx >= n_tail) return;
  const int j = n_new - n_tail + idx;
  const int64_t t = t0 + j;
  const size_t rowoff = (static_cast<size_t>(b) * n_new + j) * kDcmp;
  for (int i = lane; i < kDqk; i += 32) srow[warp][i] = in.ca[rowoff + i];
  __syncwarp();
  const size_t slot = static_cast<size_t>(b) * kWin + (t % kWin);
  warp_encode_swa(c.swa_codes + slot * (c.swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152),
                  c.swa_scales ? c.swa_scales + slot * kSwaScaleStride : nullptr, c.swa_dtype, srow[warp],
                  rope_cs + t * 64, lane);
  if (j >= n_new - 4) {
    float *dst = c.cmp_buf + (static_cast<size_t>(b) * 4 + (t & 3)) * 4 * kDcmp;
    for (int i = lane; i < kDcmp; i += 32) {
      dst[i] = in.ca[rowoff + i];
      dst[kDcmp + i] = in.cb[rowoff + i];
      dst[2 * kDcmp + i] = in.za[rowoff + i];
      dst[3 * kDcmp + i] = in.zb[rowoff + i];
    }
  }
}

// Advance n_tokens once every kernel of the append has read it.
__global__ void k_append_advance(csa2_cache c, int n_new, int64_t rope_len) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= c.batch) return;
  const int64_t t0 = c.n_tokens[b];
  if (append_ok(c, t0, n_new, rope_len)) c.n_tokens[b] = t0 + n_new;
}

}  // namespace

cudaError_t launch_kv_append(const csa2_cache &c, const void *kv, const void *ik, int in_dtype,
                             const csa2_compress_in *cmp, const float *rope_cs, int64_t rope_len, int n_new,
                             float *cmp_dbg, int32_t *err, cudaStream_t s) {
  if (n_new <= 0) return cudaSuccess;
  if (c.ratio == 1) {
    const int advance = n_new == 1 ? 1 : 0;
    k_append_r1<<<dim3(n_new, c.batch), kEncThreads, 0, s>>>(c, kv, ik, in_dtype == CSA2_IN_BF16, rope_cs, rope_len,
                                                             n_new, advance, err);
    if (advance) return cudaGetLastError();
  } else {
    const int max_emit = n_new / 2 + 1;
    dim3 g1((max_emit + kWarps - 1) / kWarps, c.batch);
    k_append_r2_entries<<<g1, 256, 0, s>>>(c, *cmp, rope_cs, rope_len, n_new, cmp_dbg, err);
    const int n_tail = n_new < kWin ? n_new : kWin;
    dim3 g2((n_tail + kWarps - 1) / kWarps, c.batch);
    k_append_r2_tail<<<g2, 256, 0, s>>>(c, *cmp, rope_cs, rope_len, n_new);
  }
  k_append_advance<<<(c.batch + 127) / 128, 128, 0, s>>>(c, n_new, rope_len);
  return cudaGetLastError();
}

}  // namespace csa2
