// csa2_select.cu -- deterministic top-k over index scores, and the candidate-pool
// build of the Hierarchical Sparse Indexer.
//
// [P5] "DeepSeek-V4: Towards Highly Efficient Million-Token Context
// Intelligence" §2.3.1: C^Sprs_t = { C_s | I_{t,s} in Top-k(I_{t,:}) }.
// [P1] "DeepSeek V4.1 Flash 아키텍처 분석" §"512개를 고르기 위해 ...": positions
// grouped 8 at a time, a block ranked by its max score, at most 2,048 blocks kept.
//
// Order: composite key K = (orderable(score) << 32) | ~slot, descending, so
// equal scores go to the lower slot (slots run in ascending position order in
// every mode); -0 == +0, NaN ranks lowest.  Every K is distinct, so the chosen
// set never depends on scheduling.
//
// Per (row, problem) -- problem 0 is the top-k over the row's slots, problem 1
// the top blocks by block maximum (FULL rows building a pool):
//   resolve  one CTA: the 13-bit histogram (from the score kernel's sideband)
//            gives the threshold bin, where the count from the top reaches k
//   collect  many CTAs: keys in bins >= the threshold go to a candidate buffer
//            (at most kSelCap; overflow is flagged)
//   final    one CTA: bitonic sort of the candidates by K, the first k kept,
//            then their positions sorted ascending and written (-1 padded).
//            After an overflow (a very crowded threshold bin) it instead runs an
//            exact radix select over the whole row.
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kChunk = 4096;  // slots per collect CTA
constexpr int kCollectThreads = 256;
constexpr int kFinalThreads = 1024;

struct SelState {
  uint32_t thr_bin;   // lowest bin that holds candidates
  uint32_t total;     // valid slots
  uint32_t ncand;     // candidates appended (may exceed kSelCap)
  uint32_t overflow;  // 1: ncand > kSelCap
};

__device__ __forceinline__ uint32_t key_of(float f) { return isnan(f) ? 0u : orderable(f); }

__device__ __forceinline__ int prob_k(const TopkArgs &a, int p) { return p == 0 ? a.k : a.out_pool_blocks; }

__device__ __forceinline__ const uint32_t *aux_hist(const uint8_t *aux, int64_t aux_row, int row, int p) {
  return reinterpret_cast<const uint32_t *>(aux + static_cast<size_t>(row) * aux_row) + static_cast<size_t>(p) * kSelBins;
}
__device__ __forceinline__ const float *aux_bmax(const uint8_t *aux, int64_t aux_row, int row) {
  return reinterpret_cast<const float *>(aux + static_cast<size_t>(row) * aux_row + 2 * kSelBins * 4);
}

// visible entries of a row
__device__ __forceinline__ int64_t row_T(const TopkArgs &a, int row) {
  int64_t T = a.q_pos[row] / a.ratio;
  return T < 0 ? 0 : T;
}

// slots of (row, problem)
__device__ __forceinline__ int64_t n_slots(const TopkArgs &a, int row, int p) {
  if (p == 1) return (min(row_T(a, row), a.stride) + 7) / 8;
  if (a.pool) return static_cast<int64_t>(a.pool_blocks) * a.bs;
  return min(row_T(a, row), a.stride);
}

// Key and output position of a slot; false if the slot is not a candidate.
__device__ __forceinline__ bool slot_key(const TopkArgs &a, const uint8_t *aux, int64_t aux_row, int row, int p,
                                         int64_t slot, int64_t T, uint32_t &key, int32_t &pos) {
  const float *sr = a.scores + static_cast<size_t>(row) * a.stride;
  if (p == 1) {
    key = key_of(aux_bmax(aux, aux_row, row)[slot]);
    pos = static_cast<int32_t>(slot);
    return true;
  }
  if (a.pool) {
    const int32_t pid = a.pool[static_cast<size_t>(row) * a.pool_blocks + slot / a.bs];
    if (pid < 0) return false;
    const int64_t q = static_cast<int64_t>(pid) * a.bs + slot % a.bs;
    if (q >= T) return false;
    pos = static_cast<int32_t>(q);
  } else {
    pos = static_cast<int32_t>(slot);
  }
  const float f = sr[slot];
  if (isnan(f)) raise_err(a.err, CSA2_DEVERR_NAN);
  key = key_of(f);
  return true;
}

// ----------------------------------------------------------------------------- sideband from scores
// grid (chunks, rows), 256 threads: histogram of the score keys, and for FULL
// rows the 8-position block maxima with their histogram.
__global__ void __launch_bounds__(256) k_fill_aux(TopkArgs a, uint8_t *aux, int64_t aux_row) {
  __shared__ uint32_t hs[kSelBins];
  const int row = blockIdx.y;
  const int64_t T = row_T(a, row);
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  const int64_t ns = n_slots(a, row, 0);
  const bool full = a.pool == nullptr;
  const int64_t nb = full ? n_slots(a, row, 1) : 0;
  if (s0 >= ns && s0 / 8 >= nb) return;
  uint32_t *gh = reinterpret_cast<uint32_t *>(aux + static_cast<size_t>(row) * aux_row);
  for (int p = 0; p < (full ? 2 : 1); ++p) {
    for (int i = threadIdx.x; i < kSelBins; i += blockDim.x) hs[i] = 0;
    __syncthreads();
    if (p == 0) {
      for (int64_t slot = s0 + threadIdx.x; slot < min(s0 + kChunk, ns); slot += blockDim.x) {
        uint32_t key;
        int32_t pos;
        if (slot_key(a, aux, aux_row, row, 0, slot, T, key, pos)) atomicAdd(&hs[key >> kSelBinShift], 1u);
      }
    } else {
      float *bm = reinterpret_cast<float *>(aux + static_cast<size_t>(row) * aux_row + 2 * kSelBins * 4);
      const float *sr = a.scores + static_cast<size_t>(row) * a.stride;
      const int64_t Tc = min(T, a.stride);
      for (int64_t b = s0 / 8 + threadIdx.x; b < min((s0 + kChunk) / 8, nb); b += blockDim.x) {
        float m = -INFINITY;
        for (int64_t q = 8 * b; q < min(8 * b + 8, Tc); ++q) m = fmaxf(m, sr[q]);
        bm[b] = m;
        atomicAdd(&hs[key_of(m) >> kSelBinShift], 1u);
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kSelBins; i += blockDim.x)
      if (hs[i]) atomicAdd(&gh[p * kSelBins + i], hs[i]);
    __syncthreads();
  }
}

// ----------------------------------------------------------------------------- resolve
// grid (rows, problems), 256 threads
__global__ void __launch_bounds__(256) k_resolve(TopkArgs a, const uint8_t *aux, int64_t aux_row, SelState *st) {
  __shared__ uint32_t warp_tot[8];
  const int row = blockIdx.x, p = blockIdx.y;
  const uint32_t *h = aux_hist(aux, aux_row, row, p);
  const int per = kSelBins / 256;  // 32 bins per thread, thread 0 owns the top bins
  uint32_t local = 0;
  for (int i = 0; i < per; ++i) local += h[kSelBins - 1 - (threadIdx.x * per + i)];
  // exclusive scan over threads (counts strictly above this thread's bins)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = local;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  uint32_t before = 0, total = 0;
  for (int w = 0; w < 8; ++w) {
    if (w < warp) before += warp_tot[w];
    total += warp_tot[w];
  }
  const uint32_t above = before + x - local;
  SelState *s = st + static_cast<size_t>(row) * 2 + p;
  const uint32_t k = static_cast<uint32_t>(prob_k(a, p));
  if (total <= k) {
    if (threadIdx.x == 0) *s = SelState{0u, total, 0u, 0u};  // every valid slot is chosen
    return;
  }
  if (above < k && k <= above + local) {
    uint32_t acc = above;
    for (int i = 0; i < per; ++i) {
      const uint32_t bin = kSelBins - 1 - (threadIdx.x * per + i);
      acc += h[bin];
      if (acc >= k) {
        *s = SelState{bin, total, 0u, 0u};
        break;
      }
    }
  }
}

// ----------------------------------------------------------------------------- collect
// grid (chunks, rows, problems), 256 threads
__global__ void __launch_bounds__(kCollectThreads) k_collect(TopkArgs a, const uint8_t *aux, int64_t aux_row,
                                                             SelState *st, uint64_t *cand) {
  const int row = blockIdx.y, p = blockIdx.z;
  const int64_t ns = n_slots(a, row, p);
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  if (s0 >= ns) return;
  SelState *s = st + static_cast<size_t>(row) * 2 + p;
  const uint32_t thr = s->thr_bin;
  const int64_t T = row_T(a, row);
  uint64_t *cb = cand + (static_cast<size_t>(row) * 2 + p) * kSelCap;
  const int lane = threadIdx.x & 31;
  for (int i = 0; i < kChunk / kCollectThreads; ++i) {
    const int64_t slot = s0 + static_cast<int64_t>(i) * kCollectThreads + threadIdx.x;
    bool want = false;
    uint64_t K = 0;
    if (slot < ns) {
      uint32_t key;
      int32_t pos;
      if (slot_key(a, aux, aux_row, row, p, slot, T, key, pos) && (key >> kSelBinShift) >= thr) {
        want = true;
        K = (static_cast<uint64_t>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(slot));
      }
    }
    const uint32_t mask = __ballot_sync(0xffffffffu, want);
    if (mask) {
      const int leader = __ffs(mask) - 1;
      uint32_t base = 0;
      if (lane == leader) base = atomicAdd(&s->ncand, static_cast<uint32_t>(__popc(mask)));
      base = __shfl_sync(0xffffffffu, base, leader);
      if (want) {
        const uint32_t at = base + __popc(mask & ((1u << lane) - 1u));
        if (at < kSelCap) cb[at] = K;
        else s->overflow = 1;
      }
    }
  }
}

// ----------------------------------------------------------------------------- final
__device__ __forceinline__ int32_t slot_position(const TopkArgs &a, int row, int p, uint32_t slot) {
  if (p == 1 || !a.pool) return static_cast<int32_t>(slot);
  const int32_t pid = a.pool[static_cast<size_t>(row) * a.pool_blocks + slot / a.bs];
  return pid * a.bs + static_cast<int32_t>(slot % a.bs);
}

// bitonic sort of n (a power of two) 64-bit keys in shared memory, descending
__device__ void bitonic_desc_u64(uint64_t *v, int n) {
  for (int size = 2; size <= n; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t x = v[lo], y = v[hi];
        if ((x < y) == desc) {
          v[lo] = y;
          v[hi] = x;
        }
      }
      __syncthreads();
    }
}
// ascending sort of n (a power of two) int32 in shared memory
__device__ void bitonic_asc_i32(int32_t *v, int n) {
  for (int size = 2; size <= n; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool asc = (lo & size) == 0;
        const int32_t x = v[lo], y = v[hi];
        if ((x > y) == asc) {
          v[lo] = y;
          v[hi] = x;
        }
      }
      __syncthreads();
    }
}

__device__ __forceinline__ int pow2_at_least(int n) {
  int m = 1;
  while (m < n) m <<= 1;
  return m;
}

// grid (rows, problems), 1024 threads; dynamic smem: kSelCap u64 + 2048 int32 + scratch
__global__ void __launch_bounds__(kFinalThreads) k_final(TopkArgs a, const uint8_t *aux, int64_t aux_row,
                                                         const SelState *st, const uint64_t *cand) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t *v = reinterpret_cast<uint64_t *>(smem);
  int32_t *pos = reinterpret_cast<int32_t *>(smem + kSelCap * 8);
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_cnt, s_prefix_hi, s_prefix_lo, s_krem;
  const int row = blockIdx.x, p = blockIdx.y;
  const SelState s = st[static_cast<size_t>(row) * 2 + p];
  const int k = prob_k(a, p);
  const int kt = static_cast<int>(min(static_cast<uint32_t>(k), s.total));  // positions to output
  int32_t *out = p == 0 ? a.idx_out + static_cast<size_t>(row) * a.k
                        : a.pool_out + static_cast<size_t>(row) * a.out_pool_blocks;

  if (!s.overflow) {
    const int n = static_cast<int>(min(s.ncand, static_cast<uint32_t>(kSelCap)));
    const int n2 = pow2_at_least(max(n, 1));
    const uint64_t *cb = cand + (static_cast<size_t>(row) * 2 + p) * kSelCap;
    for (int i = threadIdx.x; i < n2; i += blockDim.x) v[i] = i < n ? cb[i] : 0ull;
    __syncthreads();
    bitonic_desc_u64(v, n2);
    for (int i = threadIdx.x; i < kt; i += blockDim.x)
      pos[i] = slot_position(a, row, p, 0xFFFFFFFFu - static_cast<uint32_t>(v[i]));
  } else {
    // Exact radix select over the whole row: the threshold bin holds more than
    // kSelCap keys.  Find the kr-th largest K among the keys of that bin,
    // digit by digit (8 bits) over its low 51 bits, then gather.
    const int64_t ns = n_slots(a, row, p);
    const int64_t T = row_T(a, row);
    const uint32_t thr = s.thr_bin;
    if (threadIdx.x == 0) {
      s_prefix_hi = 0;
      s_prefix_lo = 0;
      s_cnt = 0;
    }
    // keys strictly above the bin
    __shared__ uint32_t s_above;
    if (threadIdx.x == 0) s_above = 0;
    __syncthreads();
    uint32_t above_local = 0;
    for (int64_t slot = threadIdx.x; slot < ns; slot += blockDim.x) {
      uint32_t key;
      int32_t q;
      if (slot_key(a, aux, aux_row, row, p, slot, T, key, q) && (key >> kSelBinShift) > thr) ++above_local;
    }
    atomicAdd(&s_above, above_local);
    __syncthreads();
    if (threadIdx.x == 0) s_krem = static_cast<uint32_t>(kt) - s_above;
    __syncthreads();
    // 51 low bits (19 score bits, then 32 slot bits), digits from the top:
    // bits 50..43, 42..35, 34..27, 26..19, 18..11, 10..3, then 2..0
    constexpr uint64_t kLow = (1ull << 51) - 1;
    uint64_t prefix = 0;
    for (int d = 0; d < 7; ++d) {
      const int sh = d < 6 ? 43 - 8 * d : 0;
      const int width = d < 6 ? 8 : 3;
      const uint64_t hi_mask = kLow & ~((1ull << (sh + width)) - 1);
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int64_t slot = threadIdx.x; slot < ns; slot += blockDim.x) {
        uint32_t key;
        int32_t q;
        if (!slot_key(a, aux, aux_row, row, p, slot, T, key, q) || (key >> kSelBinShift) != thr) continue;
        const uint64_t low = (static_cast<uint64_t>(key & ((1u << kSelBinShift) - 1)) << 32) |
                             (0xFFFFFFFFu - static_cast<uint32_t>(slot));
        if ((low & hi_mask) != (prefix & hi_mask)) continue;
        atomicAdd(&hist[(low >> sh) & ((1u << width) - 1)], 1u);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        uint32_t acc = 0;
        for (int dg = (1 << width) - 1; dg >= 0; --dg) {
          if (acc + hist[dg] >= s_krem) {
            s_krem -= acc;
            const uint64_t np_ = prefix | (static_cast<uint64_t>(dg) << sh);
            s_prefix_lo = static_cast<uint32_t>(np_);
            s_prefix_hi = static_cast<uint32_t>(np_ >> 32);
            break;
          }
          acc += hist[dg];
        }
      }
      __syncthreads();
      prefix = (static_cast<uint64_t>(s_prefix_hi) << 32) | s_prefix_lo;
    }
    // chosen: bin above thr, or in thr with low51 >= prefix (the kr-th largest)
    for (int64_t slot = threadIdx.x; slot < ns; slot += blockDim.x) {
      uint32_t key;
      int32_t q;
      if (!slot_key(a, aux, aux_row, row, p, slot, T, key, q)) continue;
      const uint32_t bin = key >> kSelBinShift;
      bool take = bin > thr;
      if (bin == thr) {
        const uint64_t low = (static_cast<uint64_t>(key & ((1u << kSelBinShift) - 1)) << 32) |
                             (0xFFFFFFFFu - static_cast<uint32_t>(slot));
        take = low >= prefix;
      }
      if (take) {
        const uint32_t at = atomicAdd(&s_cnt, 1u);
        if (at < static_cast<uint32_t>(kt)) pos[at] = q;
      }
    }
    __syncthreads();
  }
  __syncthreads();
  const int kp = pow2_at_least(max(kt, 1));
  for (int i = kt + threadIdx.x; i < kp; i += blockDim.x) pos[i] = 0x7FFFFFFF;
  __syncthreads();
  bitonic_asc_i32(pos, kp);
  const int kout = p == 0 ? a.k : a.out_pool_blocks;
  for (int i = threadIdx.x; i < kout; i += blockDim.x) out[i] = i < kt ? pos[i] : -1;
  if (p == 1 && threadIdx.x == 0) a.pool_count[row] = kt;
}

}  // namespace

size_t topk_workspace_bytes(int rows, int64_t stride, bool have_aux) {
  size_t b = static_cast<size_t>(rows) * 2 * sizeof(SelState);
  b = (b + 255) & ~size_t(255);
  b += static_cast<size_t>(rows) * 2 * kSelCap * 8;
  if (!have_aux) b += static_cast<size_t>(rows) * aux_row_bytes(stride);
  return (b + 255) & ~size_t(255);
}

cudaError_t launch_fill_aux(const TopkArgs &a, uint8_t *aux, cudaStream_t s) {
  const int64_t aux_row = aux_row_bytes(a.stride);
  cudaError_t e = cudaMemsetAsync(aux, 0, static_cast<size_t>(a.rows) * aux_row, s);
  if (e != cudaSuccess) return e;
  const int64_t slots = a.pool ? static_cast<int64_t>(a.pool_blocks) * a.bs : a.stride;
  const int chunks = static_cast<int>((slots + kChunk - 1) / kChunk);
  k_fill_aux<<<dim3(chunks > 0 ? chunks : 1, a.rows), 256, 0, s>>>(a, aux, aux_row);
  return cudaGetLastError();
}

cudaError_t launch_topk(const TopkArgs &a0, void *ws, cudaStream_t s) {
  if (a0.rows <= 0) return cudaSuccess;
  TopkArgs a = a0;
  uint8_t *w = static_cast<uint8_t *>(ws);
  SelState *st = reinterpret_cast<SelState *>(w);
  size_t off = (static_cast<size_t>(a.rows) * 2 * sizeof(SelState) + 255) & ~size_t(255);
  uint64_t *cand = reinterpret_cast<uint64_t *>(w + off);
  off += static_cast<size_t>(a.rows) * 2 * kSelCap * 8;
  const int64_t aux_row = aux_row_bytes(a.stride);
  const uint8_t *aux = a.aux;
  if (!aux) {
    uint8_t *own = w + off;
    cudaError_t e = launch_fill_aux(a, own, s);
    if (e != cudaSuccess) return e;
    aux = own;
  }
  const int nprob = (!a.pool && a.out_pool_blocks > 0) ? 2 : 1;
  const int64_t slots = a.pool ? static_cast<int64_t>(a.pool_blocks) * a.bs : a.stride;
  const int chunks = static_cast<int>((slots + kChunk - 1) / kChunk);
  k_resolve<<<dim3(a.rows, nprob), 256, 0, s>>>(a, aux, aux_row, st);
  k_collect<<<dim3(chunks > 0 ? chunks : 1, a.rows, nprob), kCollectThreads, 0, s>>>(a, aux, aux_row, st, cand);
  static bool attr = false;
  const int smem = kSelCap * 8 + 2048 * 4;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_final, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  k_final<<<dim3(a.rows, nprob), kFinalThreads, smem, s>>>(a, aux, aux_row, st, cand);
  return cudaGetLastError();
}

}  // namespace csa2
