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
//            gives the threshold bin, where the count from the top reaches k,
//            and how many keys lie strictly above it
//   collect  many CTAs: every slot whose key lies above the threshold bin is
//            chosen outright and marked in a per-row bitmap (one warp ballot per
//            32 slots writes one word); keys in the threshold bin go to a
//            candidate list (at most kSelCap; overflow is flagged)
//   final    one CTA: an exact radix select over the candidates' low 51 key
//            bits picks the ones still needed and marks them, then a block scan
//            over the bitmap writes the chosen positions in ascending order
//            (-1 padded).  After an overflow (a very crowded threshold bin) the
//            radix select runs over the whole row instead.
// Slots run in ascending position order in every mode, so the bitmap order is
// the output order and no sort is needed.
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kChunk = 4096;  // slots per collect CTA
constexpr int kCollectThreads = 256;
constexpr int kFinalThreads = 512;

struct SelState {
  uint32_t thr_bin;   // the bin where the count from the top reaches k
  uint32_t above;     // valid keys in bins above thr_bin (all chosen)
  uint32_t total;     // valid slots
  uint32_t ncand;     // keys of bin thr_bin appended (may exceed kSelCap)
  uint32_t overflow;  // 1: ncand > kSelCap
  uint32_t pad[3];
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
  __shared__ uint32_t hs[kSelBins];
  __shared__ uint32_t warp_tot[8];
  const int row = blockIdx.x, p = blockIdx.y;
  const uint4 *h4 = reinterpret_cast<const uint4 *>(aux_hist(aux, aux_row, row, p));
  for (int i = threadIdx.x; i < kSelBins / 4; i += blockDim.x) reinterpret_cast<uint4 *>(hs)[i] = h4[i];
  __syncthreads();
  // thread t owns the 32 bins kSelBins-1-32t-i, i = 0..31 (thread 0 the top ones);
  // the rotated index keeps the 32 reads of a step in distinct banks
  constexpr int per = kSelBins / 256;
  const int top = kSelBins - 1 - threadIdx.x * per;
  uint32_t local = 0;
  for (int i = 0; i < per; ++i) local += hs[top - ((i + threadIdx.x) & (per - 1))];
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
  const uint32_t above = before + x - local;  // keys in bins above this thread's
  SelState *s = st + static_cast<size_t>(row) * 2 + p;
  const uint32_t k = static_cast<uint32_t>(prob_k(a, p));
  if (total <= k) {
    // every valid slot is chosen: bin 0 is the threshold bin
    if (threadIdx.x == 0) *s = SelState{0u, total - hs[0], total, 0u, 0u, {0u, 0u, 0u}};
    return;
  }
  if (above < k && k <= above + local) {
    uint32_t acc = above;
    for (int i = 0; i < per; ++i) {
      const uint32_t bin = top - i;
      if (acc + hs[bin] >= k) {
        *s = SelState{bin, acc, total, 0u, 0u, {0u, 0u, 0u}};
        break;
      }
      acc += hs[bin];
    }
  }
}

// ----------------------------------------------------------------------------- collect
__device__ __forceinline__ uint32_t *row_bitmap(uint32_t *bm, int64_t stride, int row, int p) {
  const int64_t w0 = (stride + 31) / 32, w1 = ((stride + 7) / 8 + 31) / 32;
  return bm + static_cast<size_t>(row) * (w0 + w1) + (p ? w0 : 0);
}

// grid (chunks, rows, problems), 256 threads; thread i of a step handles slot
// s0 + 256*step + i, so warp w covers one aligned 32-slot bitmap word
__global__ void __launch_bounds__(kCollectThreads) k_collect(TopkArgs a, const uint8_t *aux, int64_t aux_row,
                                                             SelState *st, uint64_t *cand, uint32_t *bitmap) {
  constexpr int kSteps = kChunk / kCollectThreads;
  const int row = blockIdx.y, p = blockIdx.z;
  const int64_t ns = n_slots(a, row, p);
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  if (s0 >= ns) return;
  SelState *s = st + static_cast<size_t>(row) * 2 + p;
  const uint32_t thr = s->thr_bin;
  const int64_t T = row_T(a, row);
  uint64_t *cb = cand + (static_cast<size_t>(row) * 2 + p) * kSelCap;
  uint32_t *bm = row_bitmap(bitmap, a.stride, row, p);
  const int lane = threadIdx.x & 31;
  // all loads of the chunk first (independent, no side effects between them),
  // then the keys and the ballots
  float f[kSteps];
  int32_t pid[kSteps];
  const float *src = p == 1 ? aux_bmax(aux, aux_row, row) : a.scores + static_cast<size_t>(row) * a.stride;
  const bool pooled = p == 0 && a.pool != nullptr;
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int64_t slot = s0 + static_cast<int64_t>(i) * kCollectThreads + threadIdx.x;
    f[i] = slot < ns ? src[slot] : 0.0f;
    pid[i] = pooled && slot < ns ? a.pool[static_cast<size_t>(row) * a.pool_blocks + slot / a.bs] : 0;
  }
  uint32_t key[kSteps];
  uint32_t valid = 0;
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int64_t slot = s0 + static_cast<int64_t>(i) * kCollectThreads + threadIdx.x;
    bool ok = slot < ns;
    if (pooled) ok = ok && pid[i] >= 0 && static_cast<int64_t>(pid[i]) * a.bs + slot % a.bs < T;
    key[i] = key_of(f[i]);
    if (ok) valid |= 1u << i;
  }
  if (p == 0) {
#pragma unroll
    for (int i = 0; i < kSteps; ++i)
      if (((valid >> i) & 1u) && isnan(f[i])) raise_err(a.err, CSA2_DEVERR_NAN);
  }
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int64_t slot = s0 + static_cast<int64_t>(i) * kCollectThreads + threadIdx.x;
    const int64_t wbase = slot - lane;
    if (wbase >= ns) break;  // warp-uniform
    const bool ok = (valid >> i) & 1u;
    const uint32_t bin = key[i] >> kSelBinShift;
    const uint32_t word = __ballot_sync(0xffffffffu, ok && bin > thr);
    if (lane == 0) bm[wbase >> 5] = word;
    const bool want = ok && bin == thr;
    const uint32_t mask = __ballot_sync(0xffffffffu, want);
    if (mask) {
      const int leader = __ffs(mask) - 1;
      uint32_t base = 0;
      if (lane == leader) base = atomicAdd(&s->ncand, static_cast<uint32_t>(__popc(mask)));
      base = __shfl_sync(0xffffffffu, base, leader);
      if (want) {
        const uint32_t at = base + __popc(mask & ((1u << lane) - 1u));
        if (at < kSelCap)
          cb[at] = (static_cast<uint64_t>(key[i]) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(slot));
        else
          s->overflow = 1;
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

constexpr uint64_t kLow = (1ull << 51) - 1;  // key bits below the 13-bit bin: 19 score bits, 32 slot bits

__device__ __forceinline__ uint64_t low_of(uint32_t key, uint32_t slot) {
  return (static_cast<uint64_t>(key & ((1u << kSelBinShift) - 1)) << 32) | (0xFFFFFFFFu - slot);
}

// One radix digit of the select: hist holds the counts of the digit values
// among the keys that match the prefix so far; find the digit where the count
// from the top reaches *rem, extend the prefix, reduce *rem.  Warp 0 only.
__device__ __forceinline__ void pick_digit(const uint32_t *hist, int sh, uint32_t *rem, uint64_t *prefix,
                                           uint32_t *done) {
  const int lane = threadIdx.x & 31;
  uint32_t local = 0;
  for (int i = 0; i < 8; ++i) local += hist[255 - 8 * lane - i];
  uint32_t x = local;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  const uint32_t above = x - local;
  const uint32_t r = *rem;
  __syncwarp();
  if (above < r && r <= above + local) {
    uint32_t acc = above;
    for (int i = 0; i < 8; ++i) {
      const int dg = 255 - 8 * lane - i;
      if (acc + hist[dg] >= r) {
        *rem = r - acc;
        *prefix |= static_cast<uint64_t>(dg) << sh;
        // every key under this prefix is needed: the prefix (lower bits 0) is the cut
        if (hist[dg] == r - acc) *done = 1;
        break;
      }
      acc += hist[dg];
    }
  }
}

// grid (rows, problems), kFinalThreads threads; dynamic smem: kSelCap u64
__global__ void __launch_bounds__(kFinalThreads) k_final(TopkArgs a, const uint8_t *aux, int64_t aux_row,
                                                         const SelState *st, const uint64_t *cand,
                                                         uint32_t *bitmap) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t *v = reinterpret_cast<uint64_t *>(smem);
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_rem, s_done;
  __shared__ uint64_t s_prefix;
  __shared__ uint32_t warp_tot[kFinalThreads / 32];
  const int row = blockIdx.x, p = blockIdx.y;
  const SelState s = st[static_cast<size_t>(row) * 2 + p];
  const int k = prob_k(a, p);
  const uint32_t kt = min(static_cast<uint32_t>(k), s.total);  // positions to output
  const uint32_t need = kt - s.above;                           // still to choose from bin thr_bin
  const int64_t ns = n_slots(a, row, p);
  const int64_t T = row_T(a, row);
  uint32_t *bm = row_bitmap(bitmap, a.stride, row, p);
  const int n = static_cast<int>(min(s.ncand, static_cast<uint32_t>(kSelCap)));
  const bool from_row = s.overflow != 0;  // the candidates did not all fit: select over the row

  if (!from_row) {
    const uint64_t *cb = cand + (static_cast<size_t>(row) * 2 + p) * kSelCap;
    for (int i = threadIdx.x; i < n; i += blockDim.x) v[i] = cb[i];
  }
  if (threadIdx.x == 0) {
    s_rem = need;
    s_prefix = 0;
    s_done = 0;
  }
  __syncthreads();
  // exact select of the need-th largest low key among bin thr_bin: 8-bit digits
  // over bits 50..3, then bits 2..0
  const bool all = !from_row && need == static_cast<uint32_t>(n);
  if (need > 0 && !all) {
    for (int d = 0; d < 7; ++d) {
      const int sh = d < 6 ? 43 - 8 * d : 0;
      const uint32_t dmask = d < 6 ? 0xFFu : 0x7u;
      const uint64_t hi_mask = kLow & ~((1ull << (sh + (d < 6 ? 8 : 3))) - 1);
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      const uint64_t prefix = s_prefix;
      if (!from_row) {
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
          const uint64_t low = v[i] & kLow;
          if ((low & hi_mask) == prefix) atomicAdd(&hist[(low >> sh) & dmask], 1u);
        }
      } else {
        for (int64_t slot = threadIdx.x; slot < ns; slot += blockDim.x) {
          uint32_t key;
          int32_t q;
          if (!slot_key(a, aux, aux_row, row, p, slot, T, key, q) || (key >> kSelBinShift) != s.thr_bin) continue;
          const uint64_t low = low_of(key, static_cast<uint32_t>(slot));
          if ((low & hi_mask) == prefix) atomicAdd(&hist[(low >> sh) & dmask], 1u);
        }
      }
      __syncthreads();
      if (threadIdx.x < 32) pick_digit(hist, sh, &s_rem, &s_prefix, &s_done);
      __syncthreads();
      if (s_done) break;
    }
  }
  // mark the chosen keys of bin thr_bin: low >= the need-th largest
  const uint64_t cut = s_prefix;
  if (need > 0) {
    if (!from_row) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const uint64_t K = v[i];
        if (all || (K & kLow) >= cut) {
          const uint32_t slot = 0xFFFFFFFFu - static_cast<uint32_t>(K);
          atomicOr(&bm[slot >> 5], 1u << (slot & 31));
        }
      }
    } else {
      for (int64_t slot = threadIdx.x; slot < ns; slot += blockDim.x) {
        uint32_t key;
        int32_t q;
        if (!slot_key(a, aux, aux_row, row, p, slot, T, key, q) || (key >> kSelBinShift) != s.thr_bin) continue;
        if (low_of(key, static_cast<uint32_t>(slot)) >= cut) atomicOr(&bm[slot >> 5], 1u << (slot & 31));
      }
    }
  }
  __syncthreads();
  // ascending output: block scan of the bitmap's popcounts
  const int64_t nw = (ns + 31) / 32;
  const int64_t per = (nw + blockDim.x - 1) / blockDim.x;
  const int64_t w0 = threadIdx.x * per, w1 = min(nw, w0 + per);
  uint32_t cnt = 0;
  for (int64_t w = w0; w < w1; ++w) cnt += __popc(bm[w]);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  uint32_t off = x - cnt;
  for (int w = 0; w < warp; ++w) off += warp_tot[w];
  int32_t *out = p == 0 ? a.idx_out + static_cast<size_t>(row) * a.k
                        : a.pool_out + static_cast<size_t>(row) * a.out_pool_blocks;
  for (int64_t w = w0; w < w1; ++w) {
    uint32_t word = bm[w];
    while (word) {
      const int b = __ffs(word) - 1;
      word &= word - 1;
      if (off < kt) out[off] = slot_position(a, row, p, static_cast<uint32_t>(w * 32 + b));
      ++off;
    }
  }
  const int kout = p == 0 ? a.k : a.out_pool_blocks;
  for (int i = kt + threadIdx.x; i < kout; i += blockDim.x) out[i] = -1;
  if (p == 1 && threadIdx.x == 0) a.pool_count[row] = static_cast<int32_t>(kt);
}

}  // namespace

// Workspace: selection state | candidates | bitmaps | (sideband, when the
// caller has none)
size_t topk_workspace_bytes(int rows, int64_t stride, bool have_aux) {
  size_t b = static_cast<size_t>(rows) * 2 * sizeof(SelState);
  b = (b + 255) & ~size_t(255);
  b += static_cast<size_t>(rows) * 2 * kSelCap * 8;
  const int64_t w0 = (stride + 31) / 32, w1 = ((stride + 7) / 8 + 31) / 32;
  b += (static_cast<size_t>(rows) * (w0 + w1) * 4 + 255) & ~size_t(255);
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
  uint32_t *bitmap = reinterpret_cast<uint32_t *>(w + off);
  const int64_t w0 = (a.stride + 31) / 32, w1 = ((a.stride + 7) / 8 + 31) / 32;
  off += (static_cast<size_t>(a.rows) * (w0 + w1) * 4 + 255) & ~size_t(255);
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
  k_collect<<<dim3(chunks > 0 ? chunks : 1, a.rows, nprob), kCollectThreads, 0, s>>>(a, aux, aux_row, st, cand,
                                                                                     bitmap);
  const int smem = kSelCap * 8;
  k_final<<<dim3(a.rows, nprob), kFinalThreads, smem, s>>>(a, aux, aux_row, st, cand, bitmap);
  return cudaGetLastError();
}

}  // namespace csa2
