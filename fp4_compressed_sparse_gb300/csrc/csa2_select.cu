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
// One thread-block cluster of 4 or 8 CTAs (512 threads each) per (row, problem)
// -- problem 0 is the top-k over the row's slots, problem 1 the top blocks by
// block maximum (FULL rows building a pool).  Each CTA of the cluster owns a
// contiguous slice of the row's bitmap words, in shared memory (in the
// workspace when a slice exceeds 128 KB):
//   1. every CTA reads the row's 13-bit key histogram (the score kernel's
//      sideband) and finds the threshold bin, where the count from the top
//      reaches k, and how many keys lie strictly above it;
//   2. one pass over its slice of the row (just written, so mostly from L2): a
//      slot whose key lies above the threshold bin is chosen outright and marked
//      in the slice's bitmap (one warp ballot per 32 slots writes one word);
//      keys in the threshold bin go to the CTA's candidate list;
//   3. after a cluster barrier the leader CTA gathers every candidate list
//      through distributed shared memory, runs an exact radix select over the
//      candidates' low 51 key bits and marks the ones still needed in their
//      owners' slices (after an overflow of the lists it runs over the row);
//   4. each CTA scans its slice's popcounts, offsets them by the lower slices'
//      counts and writes the chosen positions in ascending order, -1 padded.
// Slots run in ascending position order in every mode, so the bitmap order is
// the output order and no sort is needed.
// Launches with more (row, problem) pairs than one wave of such clusters holds
// (the chunked prefill's query blocks) run k_select_row instead: the same steps
// inside one 1024-thread CTA per (row, problem).
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kChunk = 4096;  // slots per sideband-fill CTA
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelClusterMax = 8;            // CTAs per (row, problem), one cluster sharing the row: 4 or 8
constexpr int64_t kSmemBitmapWords = 32768;  // a CTA's bitmap slice stays in shared memory up to 128 KB

__device__ __forceinline__ uint32_t key_of(float f) { return isnan(f) ? 0u : orderable(f); }

// The float whose order key is k (k >= 1; the inverse of orderable()).
__device__ __forceinline__ float float_of_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// The lowest non-NaN value of histogram bin b > 0.  Keys below that of -inf
// (0x007FFFFF) belong to negative NaN payloads, which rank as key 0: the bin
// holding -inf starts at -inf, not at the NaN its first key decodes to.
__device__ __forceinline__ float bin_low(uint32_t b) {
  const uint32_t k = b << kSelBinShift;
  return float_of_key(k > 0x007FFFFFu ? k : 0x007FFFFFu);
}
// The highest non-NaN value of bin b: keys above that of +inf (0xFF800000)
// belong to positive NaN payloads.
__device__ __forceinline__ float bin_high(uint32_t b) {
  const uint32_t k = ((b + 1) << kSelBinShift) - 1;
  return float_of_key(k < 0xFF800000u ? k : 0xFF800000u);
}

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

// ----------------------------------------------------------------------------- select
__device__ __forceinline__ int32_t slot_position(const TopkArgs &a, int row, int p, uint32_t slot) {
  if (p == 1 || !a.pool) return static_cast<int32_t>(slot);
  const int32_t pid = a.pool[static_cast<size_t>(row) * a.pool_blocks + slot / a.bs];
  return pid * a.bs + static_cast<int32_t>(slot % a.bs);
}

constexpr uint64_t kLow = (1ull << 51) - 1;  // key bits below the 13-bit bin: 19 score bits, 32 slot bits

__device__ __forceinline__ uint64_t low_of(uint32_t key, uint32_t slot) {
  return (static_cast<uint64_t>(key & ((1u << kSelBinShift) - 1)) << 32) | (0xFFFFFFFFu - slot);
}

__device__ __forceinline__ uint32_t *row_bitmap(uint32_t *bm, int64_t stride, int row, int p) {
  const int64_t w0 = (stride + 31) / 32, w1 = ((stride + 7) / 8 + 31) / 32;
  return bm + static_cast<size_t>(row) * (w0 + w1) + (p ? w0 : 0);
}

// Block-wide exclusive scan of one value per thread; *total = the sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_tot, uint32_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < kSelWarps ? warp_tot[lane] : 0u, inc = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane < kSelWarps) warp_tot[lane] = inc - t;  // exclusive warp offsets
    if (lane == kSelWarps - 1) warp_tot[kSelWarps] = inc;
  }
  __syncthreads();
  const uint32_t r = warp_tot[warp] + x - v;
  *total = warp_tot[kSelWarps];
  __syncthreads();  // warp_tot may be reused right away
  return r;
}

// One radix digit of the select (warp 0): hist holds the counts of the digit
// values among the keys matching the prefix so far; find the digit where the
// count from the top reaches *rem, extend the prefix, reduce *rem; *done when
// every key under the new prefix is needed.
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
        if (hist[dg] == r - acc) *done = 1;
        break;
      }
      acc += hist[dg];
    }
  }
}

struct SelSmem {
  uint64_t cand[kSelCap];  // this CTA's keys of the threshold bin; the leader then gathers everyone's
  uint32_t warp_tot[kSelWarps + 1];
  uint32_t dhist[256];
  uint64_t prefix;
  uint32_t thr, above, total, ncand, overflow, rem, done;
  uint32_t cnt_below;  // chosen slots in the lower-ranked slices (their CTAs add to it)
};

// Key of slot `slot` (valid only when *ok): reads of one warp step go to 32
// consecutive slots.
__device__ __forceinline__ float slot_value(const TopkArgs &a, const float *src, const int32_t *prow, int p,
                                            int64_t slot, int64_t ns, int64_t T, bool &ok) {
  ok = slot < ns;
  if (!ok) return 0.0f;
  if (p == 0 && a.pool) {
    const int32_t pid = prow[slot / a.bs];
    ok = pid >= 0 && static_cast<int64_t>(pid) * a.bs + slot % a.bs < T;
  }
  return src[slot];
}

// ---- distributed shared memory (the CTAs of one cluster)
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(const void *p, uint32_t rank) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(dsmem_addr(p, rank)) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_dsmem_u64(const void *p, uint32_t rank) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];\n" : "=l"(v) : "r"(dsmem_addr(p, rank)) : "memory");
  return v;
}
__device__ __forceinline__ void or_dsmem(uint32_t *p, uint32_t rank, uint32_t v) {
  asm volatile("red.shared::cluster.or.b32 [%0], %1;\n" ::"r"(dsmem_addr(p, rank)), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// bitmap words of one cluster CTA: a multiple of 4 (the vector pass takes 4 words per step)
__host__ __device__ __forceinline__ int64_t span_words(int64_t nw, int ncl) {
  return ((nw + ncl - 1) / ncl + 3) / 4 * 4;
}

// grid (ncl, rows, problems), cluster (ncl, 1, 1), kSelThreads;
// dynamic smem: SelSmem + this CTA's bitmap slice (when it fits)
__global__ void __launch_bounds__(kSelThreads, 2) k_select(TopkArgs a, const uint8_t *aux, int64_t aux_row,
                                                           uint32_t *bitmap_g, int bitmap_in_smem, int ncl) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem &sm = *reinterpret_cast<SelSmem *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = blockIdx.x;  // rank in the cluster
  const int row = blockIdx.y, p = blockIdx.z;
  const int64_t ns = n_slots(a, row, p);
  const int64_t T = row_T(a, row);
  const uint32_t k = static_cast<uint32_t>(prob_k(a, p));
  const int64_t nw = (ns + 31) / 32;
  const int64_t span = span_words(nw, ncl);
  const int64_t w_lo = min(nw, static_cast<int64_t>(rank) * span), w_hi = min(nw, w_lo + span);
  uint32_t *bm_local = bitmap_in_smem ? reinterpret_cast<uint32_t *>(smem_raw + sizeof(SelSmem))
                                      : row_bitmap(bitmap_g, a.stride, row, p) + w_lo;
  // word w of the row lives in CTA w / span at offset w % span
  const float *src = p == 1 ? aux_bmax(aux, aux_row, row) : a.scores + static_cast<size_t>(row) * a.stride;
  const int32_t *prow = a.pool ? a.pool + static_cast<size_t>(row) * a.pool_blocks : nullptr;

  // the first batch of the streaming pass does not depend on the threshold:
  // request it now (FULL rows and block maxima)
  constexpr int kFB = 16;  // words per warp per batch in the fast pass
  const bool plain = p == 1 || a.pool == nullptr;
  const uint32_t nsu = static_cast<uint32_t>(ns);
  float fb[kFB];
  if (plain) {
#pragma unroll
    for (int b = 0; b < kFB; ++b) {
      const int64_t w = w_lo + static_cast<int64_t>(warp) * kFB + b;
      const uint32_t slot = static_cast<uint32_t>(w * 32 + lane);
      fb[b] = (w < w_hi && slot < nsu) ? src[slot] : __uint_as_float(0x7FC00000u);
    }
  }

  // ---- 1. threshold bin from the histogram (every CTA of the cluster, identically)
  {
    // thread t owns the bins kSelBins-1-per*t-i (thread 0 the top ones): per
    // contiguous, 16-byte aligned counts, read straight into registers
    constexpr int per = kSelBins / kSelThreads;
    const int top = kSelBins - 1 - tid * per;
    const uint32_t base = static_cast<uint32_t>(top - per + 1);  // hb[j] = count of bin base + j
    uint32_t hb[per];
    const uint4 *h4 = reinterpret_cast<const uint4 *>(aux_hist(aux, aux_row, row, p)) + base / 4;
#pragma unroll
    for (int q = 0; q < per / 4; ++q) {
      const uint4 v = h4[q];
      hb[4 * q] = v.x;
      hb[4 * q + 1] = v.y;
      hb[4 * q + 2] = v.z;
      hb[4 * q + 3] = v.w;
    }
    if (tid == 0) {
      sm.ncand = 0;
      sm.cnt_below = 0;
      sm.overflow = 0;
      sm.rem = 0;
      sm.done = 0;
      sm.prefix = 0;
    }
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) local += hb[j];
    uint32_t total;
    const uint32_t above = block_excl_scan(local, sm.warp_tot, &total);  // also orders the writes above
    if (total <= k) {
      if (base == 0) {  // the owner of bin 0: every valid slot is chosen, bin 0 is the threshold bin
        sm.thr = 0;
        sm.above = total - hb[0];
        sm.total = total;
      }
    } else if (above < k && k <= above + local) {
      uint32_t acc = above;
      bool found = false;
#pragma unroll
      for (int i = 0; i < per; ++i) {
        const uint32_t c = hb[per - 1 - i];  // bin top - i
        if (!found && acc + c >= k) {
          sm.thr = static_cast<uint32_t>(top - i);
          sm.above = acc;
          sm.total = total;
          found = true;
        }
        acc += c;
      }
    }
    __syncthreads();
  }
  const uint32_t thr = sm.thr;
  const uint32_t kt = min(k, sm.total);
  const uint32_t need = kt - sm.above;

  // ---- 2. one pass over this CTA's words: bitmap words of the keys above the
  // bin, candidates in it
  auto add_cands = [&](uint32_t mask, bool want, uint64_t K) {
    if (!mask) return;
    const int leader = __ffs(mask) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(&sm.ncand, static_cast<uint32_t>(__popc(mask)));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (want) {
      const uint32_t at = base + __popc(mask & ((1u << lane) - 1u));
      if (at < kSelCap) sm.cand[at] = K;
      else sm.overflow = 1;
    }
  };
  if (plain && thr > 0) {
    // order keys are monotone in the float value: "above the bin" is f > hi and
    // "in the bin" is lo <= f <= hi (exact, -0 == +0; NaN is neither, like its
    // key 0 when the threshold bin is above 0); slots outside the row read as NaN
    const float lo = bin_low(thr);
    const float hi = bin_high(thr);
    bool nan_seen = false;  // a NaN score in this lane's slots (reported once, after the pass)
    for (int64_t w0 = w_lo + static_cast<int64_t>(warp) * kFB; w0 < w_hi; w0 += static_cast<int64_t>(kSelWarps) * kFB) {
      if (w0 != w_lo + static_cast<int64_t>(warp) * kFB) {
#pragma unroll
        for (int b = 0; b < kFB; ++b) {
          const int64_t w = w0 + b;
          const uint32_t slot = static_cast<uint32_t>(w * 32 + lane);
          fb[b] = (w < w_hi && slot < nsu) ? src[slot] : __uint_as_float(0x7FC00000u);
        }
      }
#pragma unroll
      for (int b = 0; b < kFB; ++b) {
        const int64_t w = w0 + b;
        if (w >= w_hi) break;  // warp-uniform
        const float f = fb[b];
        const uint32_t slot = static_cast<uint32_t>(w * 32 + lane);
        nan_seen |= isnan(f) && slot < nsu;
        const uint32_t word = __ballot_sync(0xffffffffu, f > hi);
        if (lane == 0) bm_local[w - w_lo] = word;
        const bool want = f >= lo && f <= hi;
        const uint32_t mask = __ballot_sync(0xffffffffu, want);
        if (mask)  // the candidate keys only where a word has any
          add_cands(mask, want, (static_cast<uint64_t>(orderable(f)) << 32) | (0xFFFFFFFFu - slot));
      }
    }
    if (p == 0 && nan_seen) raise_err(a.err, CSA2_DEVERR_NAN);
  } else {
    for (int64_t w = w_lo + warp; w < w_hi; w += kSelWarps) {
      bool ok;
      const int64_t slot = w * 32 + lane;
      const float f = slot_value(a, src, prow, p, slot, ns, T, ok);
      if (p == 0 && ok && isnan(f)) raise_err(a.err, CSA2_DEVERR_NAN);
      const uint32_t key = key_of(f);
      const uint32_t bin = key >> kSelBinShift;
      const uint32_t word = __ballot_sync(0xffffffffu, ok && bin > thr);
      if (lane == 0) bm_local[w - w_lo] = word;
      const bool want = ok && bin == thr;
      add_cands(__ballot_sync(0xffffffffu, want), want,
                (static_cast<uint64_t>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(slot)));
    }
  }
  cluster_sync();  // #1: every slice and candidate list complete

  // ---- 3. the leader gathers the candidates and selects the ones still needed
  if (rank == 0) {
    // every peer's count and overflow flag, then every peer's candidates, are
    // requested before any of them is used: two round trips in all
    uint32_t cnt[kSelClusterMax], off[kSelClusterMax], ovr[kSelClusterMax], n = 0, ovf = sm.overflow, maxc = 0;
    cnt[0] = sm.ncand;
#pragma unroll
    for (int r = 1; r < kSelClusterMax; ++r) {
      cnt[r] = 0;
      ovr[r] = 0;
      if (r < ncl) {
        cnt[r] = ld_dsmem_u32(&sm.ncand, r);
        ovr[r] = ld_dsmem_u32(&sm.overflow, r);
      }
    }
#pragma unroll
    for (int r = 0; r < kSelClusterMax; ++r) {
      if (r > 0) {
        ovf |= ovr[r];
        maxc = max(maxc, cnt[r]);
      }
      off[r] = n;
      n += cnt[r];
    }
    const bool from_row = ovf != 0 || n > static_cast<uint32_t>(kSelCap);
    if (!from_row) {
      for (uint32_t i = tid; i < maxc; i += kSelThreads) {
        uint64_t v[kSelClusterMax];
#pragma unroll
        for (int r = 1; r < kSelClusterMax; ++r)
          if (i < cnt[r]) v[r] = ld_dsmem_u64(&sm.cand[i], r);
#pragma unroll
        for (int r = 1; r < kSelClusterMax; ++r)
          if (i < cnt[r]) sm.cand[off[r] + i] = v[r];
      }
    }
    __syncthreads();
    if (tid == 0) sm.rem = need;
    __syncthreads();
    // exact select of the need-th largest low key in the bin: 8-bit digits over
    // bits 50..3, then bits 2..0
    const int nc = static_cast<int>(n);
    const bool all = !from_row && need == n;
    if (need > 0 && !all) {
      for (int d = 0; d < 7; ++d) {
        const int sh = d < 6 ? 43 - 8 * d : 0;
        const uint32_t dmask = d < 6 ? 0xFFu : 0x7u;
        const uint64_t hi_mask = kLow & ~((1ull << (sh + (d < 6 ? 8 : 3))) - 1);
        for (int i = tid; i < 256; i += kSelThreads) sm.dhist[i] = 0;
        __syncthreads();
        const uint64_t prefix = sm.prefix;
        if (!from_row) {
          for (int i = tid; i < nc; i += kSelThreads) {
            const uint64_t low = sm.cand[i] & kLow;
            if ((low & hi_mask) == prefix) atomicAdd(&sm.dhist[(low >> sh) & dmask], 1u);
          }
        } else {
          for (int64_t slot = tid; slot < ns; slot += kSelThreads) {
            bool ok;
            const float f = slot_value(a, src, prow, p, slot, ns, T, ok);
            const uint32_t key = key_of(f);
            if (!ok || (key >> kSelBinShift) != thr) continue;
            const uint64_t low = low_of(key, static_cast<uint32_t>(slot));
            if ((low & hi_mask) == prefix) atomicAdd(&sm.dhist[(low >> sh) & dmask], 1u);
          }
        }
        __syncthreads();
        if (warp == 0) pick_digit(sm.dhist, sh, &sm.rem, &sm.prefix, &sm.done);
        __syncthreads();
        if (sm.done) break;
      }
    }
    // mark the chosen keys of the bin (low >= the need-th largest) in their owners' slices
    const uint64_t cut = sm.prefix;
    auto mark = [&](uint32_t slot) {
      const int64_t w = slot >> 5;
      const uint32_t owner = static_cast<uint32_t>(w / span);
      const uint32_t bit = 1u << (slot & 31);
      if (bitmap_in_smem) or_dsmem(reinterpret_cast<uint32_t *>(smem_raw + sizeof(SelSmem)) + (w - owner * span), owner, bit);
      else atomicOr(row_bitmap(bitmap_g, a.stride, row, p) + w, bit);
    };
    if (need > 0) {
      if (!from_row) {
        for (int i = tid; i < nc; i += kSelThreads) {
          const uint64_t K = sm.cand[i];
          if (all || (K & kLow) >= cut) mark(0xFFFFFFFFu - static_cast<uint32_t>(K));
        }
      } else {
        for (int64_t slot = tid; slot < ns; slot += kSelThreads) {
          bool ok;
          const float f = slot_value(a, src, prow, p, slot, ns, T, ok);
          const uint32_t key = key_of(f);
          if (!ok || (key >> kSelBinShift) != thr) continue;
          if (low_of(key, static_cast<uint32_t>(slot)) >= cut) mark(static_cast<uint32_t>(slot));
        }
      }
    }
  }
  cluster_sync();  // #2: every chosen slot is marked

  // ---- 4. ascending output: block scan of this slice's popcounts, offset by
  // the counts of the lower-ranked slices
  const int64_t nloc = w_hi - w_lo;
  const int64_t per = (nloc + kSelThreads - 1) / kSelThreads;
  const int64_t wb = min(nloc, tid * per), we = min(nloc, wb + per);
  uint32_t c = 0;
  for (int64_t w = wb; w < we; ++w) c += __popc(bm_local[w]);
  uint32_t tot;
  uint32_t off = block_excl_scan(c, sm.warp_tot, &tot);
  // every higher-ranked slice starts after this one: add this slice's count to
  // theirs (cnt_below was cleared before barrier #1)
  if (tid > 0 && tid < ncl && static_cast<uint32_t>(tid) > rank)
    asm volatile("red.shared::cluster.add.u32 [%0], %1;\n" ::"r"(dsmem_addr(&sm.cnt_below, tid)), "r"(tot) : "memory");
  cluster_sync();  // #3: every slice's count added; no shared memory of a peer is touched after it
  off += sm.cnt_below;
  int32_t *out = p == 0 ? a.idx_out + static_cast<size_t>(row) * a.k
                        : a.pool_out + static_cast<size_t>(row) * a.out_pool_blocks;
  for (int64_t w = wb; w < we; ++w) {
    uint32_t word = bm_local[w];
    while (word) {
      const int b = __ffs(word) - 1;
      word &= word - 1;
      if (off < kt) out[off] = slot_position(a, row, p, static_cast<uint32_t>((w_lo + w) * 32 + b));
      ++off;
    }
  }
  if (rank == static_cast<uint32_t>(ncl) - 1) {
    const int kout = p == 0 ? a.k : a.out_pool_blocks;
    for (int i = kt + tid; i < kout; i += kSelThreads) out[i] = -1;
    if (p == 1 && tid == 0) a.pool_count[row] = static_cast<int32_t>(kt);
  }
}

// ----------------------------------------------------------------------------- one CTA per row
// Many rows of at most kRowMaxSlots slots (the chunked prefill's query rows):
// one CTA of 1024 threads per (row, problem), no cluster, so that the launch
// needs a quarter of the CTAs (and waves) of the cluster kernel.  The same
// selection as k_select with every step inside one CTA: threshold bin from the
// sideband histogram, one pass over the row (bitmap of the keys above the bin,
// candidate list of the keys in it), exact radix select among the candidates
// (or over the row after a list overflow), then the ascending output from a
// block scan of the bitmap's popcounts.
constexpr int kRowThreads = 1024;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int64_t kRowMaxSlots = 131072;
constexpr int kRowMaxWords = static_cast<int>(kRowMaxSlots / 32);

struct RowSmem {
  uint64_t cand[kSelCap];
  uint32_t bitmap[kRowMaxWords];
  uint32_t warp_tot[kRowWarps + 1];
  uint32_t dhist[256];
  uint64_t prefix;
  uint32_t thr, above, total, ncand, overflow, rem, done;
};

// Block-wide exclusive scan over kRowThreads threads; *total = the sum.
__device__ __forceinline__ uint32_t row_excl_scan(uint32_t v, uint32_t *warp_tot, uint32_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const uint32_t t = warp_tot[lane];
    uint32_t inc = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    warp_tot[lane] = inc - t;  // exclusive warp offsets
    if (lane == 31) warp_tot[kRowWarps] = inc;
  }
  __syncthreads();
  const uint32_t r = warp_tot[warp] + x - v;
  *total = warp_tot[kRowWarps];
  __syncthreads();  // warp_tot may be reused right away
  return r;
}

// grid (rows, problems), kRowThreads; dynamic smem: RowSmem
__global__ void __launch_bounds__(kRowThreads, 1) k_select_row(TopkArgs a, const uint8_t *aux, int64_t aux_row) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RowSmem &sm = *reinterpret_cast<RowSmem *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x, p = blockIdx.y;
  const int64_t ns = n_slots(a, row, p);
  const int64_t T = row_T(a, row);
  const uint32_t k = static_cast<uint32_t>(prob_k(a, p));
  const int nw = static_cast<int>((ns + 31) / 32);
  const float *src = p == 1 ? aux_bmax(aux, aux_row, row) : a.scores + static_cast<size_t>(row) * a.stride;
  const int32_t *prow = a.pool ? a.pool + static_cast<size_t>(row) * a.pool_blocks : nullptr;
  const bool plain = p == 1 || a.pool == nullptr;
  const uint32_t nsu = static_cast<uint32_t>(ns);

  // the first batch of the pass does not depend on the threshold: request it now
  constexpr int kFB = 16;  // words per warp per batch
  float fb[kFB];
  if (plain) {
#pragma unroll
    for (int b = 0; b < kFB; ++b) {
      const int w = warp * kFB + b;
      const uint32_t slot = static_cast<uint32_t>(w) * 32 + lane;
      fb[b] = (w < nw && slot < nsu) ? src[slot] : __uint_as_float(0x7FC00000u);
    }
  }

  // ---- 1. threshold bin from the histogram
  {
    constexpr int per = kSelBins / kRowThreads;  // 8 contiguous bins per thread, thread 0 the top ones
    const int top = kSelBins - 1 - tid * per;
    const uint32_t base = static_cast<uint32_t>(top - per + 1);  // hb[j] = count of bin base + j
    uint32_t hb[per];
    const uint4 *h4 = reinterpret_cast<const uint4 *>(aux_hist(aux, aux_row, row, p)) + base / 4;
#pragma unroll
    for (int q = 0; q < per / 4; ++q) {
      const uint4 v = h4[q];
      hb[4 * q] = v.x;
      hb[4 * q + 1] = v.y;
      hb[4 * q + 2] = v.z;
      hb[4 * q + 3] = v.w;
    }
    for (int i = tid; i < nw; i += kRowThreads) sm.bitmap[i] = 0;
    if (tid == 0) {
      sm.ncand = 0;
      sm.overflow = 0;
      sm.rem = 0;
      sm.done = 0;
      sm.prefix = 0;
    }
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) local += hb[j];
    uint32_t total;
    const uint32_t above = row_excl_scan(local, sm.warp_tot, &total);  // also orders the writes above
    if (total <= k) {
      if (base == 0) {  // the owner of bin 0: every valid slot is chosen, bin 0 is the threshold bin
        sm.thr = 0;
        sm.above = total - hb[0];
        sm.total = total;
      }
    } else if (above < k && k <= above + local) {
      uint32_t acc = above;
      bool found = false;
#pragma unroll
      for (int i = 0; i < per; ++i) {
        const uint32_t c = hb[per - 1 - i];  // bin top - i
        if (!found && acc + c >= k) {
          sm.thr = static_cast<uint32_t>(top - i);
          sm.above = acc;
          sm.total = total;
          found = true;
        }
        acc += c;
      }
    }
    __syncthreads();
  }
  const uint32_t thr = sm.thr;
  const uint32_t kt = min(k, sm.total);
  const uint32_t need = kt - sm.above;

  // ---- 2. one pass over the row: bitmap words of the keys above the bin,
  // candidates in it
  auto add_cands = [&](uint32_t mask, bool want, uint64_t K) {
    if (!mask) return;
    const int leader = __ffs(mask) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(&sm.ncand, static_cast<uint32_t>(__popc(mask)));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (want) {
      const uint32_t at = base + __popc(mask & ((1u << lane) - 1u));
      if (at < kSelCap) sm.cand[at] = K;
      else sm.overflow = 1;
    }
  };
  if (plain && thr > 0) {
    // "above the bin" is f > hi and "in the bin" lo <= f <= hi (order keys are
    // monotone in the float value; -0 == +0; NaN is neither)
    const float lo = bin_low(thr);
    const float hi = bin_high(thr);
    bool nan_seen = false;  // a NaN score in this lane's slots (reported once, after the pass)
    for (int w0 = warp * kFB; w0 < nw; w0 += kRowWarps * kFB) {
      if (w0 != warp * kFB) {
#pragma unroll
        for (int b = 0; b < kFB; ++b) {
          const int w = w0 + b;
          const uint32_t slot = static_cast<uint32_t>(w) * 32 + lane;
          fb[b] = (w < nw && slot < nsu) ? src[slot] : __uint_as_float(0x7FC00000u);
        }
      }
#pragma unroll
      for (int b = 0; b < kFB; ++b) {
        const int w = w0 + b;
        if (w >= nw) break;  // warp-uniform
        const float f = fb[b];
        const uint32_t slot = static_cast<uint32_t>(w) * 32 + lane;
        nan_seen |= isnan(f) && slot < nsu;
        const uint32_t word = __ballot_sync(0xffffffffu, f > hi);
        if (lane == 0) sm.bitmap[w] = word;
        const bool want = f >= lo && f <= hi;
        const uint32_t mask = __ballot_sync(0xffffffffu, want);
        if (mask)  // the candidate keys only where a word has any
          add_cands(mask, want, (static_cast<uint64_t>(orderable(f)) << 32) | (0xFFFFFFFFu - slot));
      }
    }
    if (p == 0 && nan_seen) raise_err(a.err, CSA2_DEVERR_NAN);
  } else {
    for (int w = warp; w < nw; w += kRowWarps) {
      bool ok;
      const int64_t slot = static_cast<int64_t>(w) * 32 + lane;
      const float f = slot_value(a, src, prow, p, slot, ns, T, ok);
      if (p == 0 && ok && isnan(f)) raise_err(a.err, CSA2_DEVERR_NAN);
      const uint32_t key = key_of(f);
      const uint32_t bin = key >> kSelBinShift;
      const uint32_t word = __ballot_sync(0xffffffffu, ok && bin > thr);
      if (lane == 0) sm.bitmap[w] = word;
      const bool want = ok && bin == thr;
      add_cands(__ballot_sync(0xffffffffu, want), want,
                (static_cast<uint64_t>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(slot)));
    }
  }
  __syncthreads();

  // ---- 3. exact select of the need-th largest low key in the bin: 8-bit
  // digits over bits 50..3, then bits 2..0 (over the row after a list overflow)
  const uint32_t n = sm.ncand;
  const bool from_row = sm.overflow != 0 || n > static_cast<uint32_t>(kSelCap);
  const int nc = static_cast<int>(n);
  const bool all = !from_row && need == n;
  if (tid == 0) sm.rem = need;
  __syncthreads();
  if (need > 0 && !all) {
    for (int d = 0; d < 7; ++d) {
      const int sh = d < 6 ? 43 - 8 * d : 0;
      const uint32_t dmask = d < 6 ? 0xFFu : 0x7u;
      const uint64_t hi_mask = kLow & ~((1ull << (sh + (d < 6 ? 8 : 3))) - 1);
      for (int i = tid; i < 256; i += kRowThreads) sm.dhist[i] = 0;
      __syncthreads();
      const uint64_t prefix = sm.prefix;
      if (!from_row) {
        for (int i = tid; i < nc; i += kRowThreads) {
          const uint64_t low = sm.cand[i] & kLow;
          if ((low & hi_mask) == prefix) atomicAdd(&sm.dhist[(low >> sh) & dmask], 1u);
        }
      } else {
        for (int64_t slot = tid; slot < ns; slot += kRowThreads) {
          bool ok;
          const float f = slot_value(a, src, prow, p, slot, ns, T, ok);
          const uint32_t key = key_of(f);
          if (!ok || (key >> kSelBinShift) != thr) continue;
          const uint64_t low = low_of(key, static_cast<uint32_t>(slot));
          if ((low & hi_mask) == prefix) atomicAdd(&sm.dhist[(low >> sh) & dmask], 1u);
        }
      }
      __syncthreads();
      if (warp == 0) pick_digit(sm.dhist, sh, &sm.rem, &sm.prefix, &sm.done);
      __syncthreads();
      if (sm.done) break;
    }
  }
  // mark the chosen keys of the bin (low >= the need-th largest)
  const uint64_t cut = sm.prefix;
  if (need > 0) {
    if (!from_row) {
      for (int i = tid; i < nc; i += kRowThreads) {
        const uint64_t K = sm.cand[i];
        if (all || (K & kLow) >= cut) {
          const uint32_t slot = 0xFFFFFFFFu - static_cast<uint32_t>(K);
          atomicOr(&sm.bitmap[slot >> 5], 1u << (slot & 31));
        }
      }
    } else {
      for (int64_t slot = tid; slot < ns; slot += kRowThreads) {
        bool ok;
        const float f = slot_value(a, src, prow, p, slot, ns, T, ok);
        const uint32_t key = key_of(f);
        if (!ok || (key >> kSelBinShift) != thr) continue;
        if (low_of(key, static_cast<uint32_t>(slot)) >= cut)
          atomicOr(&sm.bitmap[slot >> 5], 1u << (static_cast<uint32_t>(slot) & 31));
      }
    }
  }
  __syncthreads();

  // ---- 4. ascending output: block scan of the popcounts of contiguous word ranges
  const int per = (nw + kRowThreads - 1) / kRowThreads;
  const int wb = min(nw, tid * per), we = min(nw, wb + per);
  uint32_t c = 0;
  for (int w = wb; w < we; ++w) c += __popc(sm.bitmap[w]);
  uint32_t tot;
  uint32_t off = row_excl_scan(c, sm.warp_tot, &tot);
  int32_t *out = p == 0 ? a.idx_out + static_cast<size_t>(row) * a.k
                        : a.pool_out + static_cast<size_t>(row) * a.out_pool_blocks;
  for (int w = wb; w < we; ++w) {
    uint32_t word = sm.bitmap[w];
    while (word) {
      const int b = __ffs(word) - 1;
      word &= word - 1;
      if (off < kt) out[off] = slot_position(a, row, p, static_cast<uint32_t>(w) * 32 + b);
      ++off;
    }
  }
  const int kout = p == 0 ? a.k : a.out_pool_blocks;
  for (int i = kt + tid; i < kout; i += kRowThreads) out[i] = -1;
  if (p == 1 && tid == 0) a.pool_count[row] = static_cast<int32_t>(kt);
}

}  // namespace

// Workspace: bitmaps (used when a row has more than 2^20 slots) | the
// sideband, when the caller has none
size_t topk_workspace_bytes(int rows, int64_t stride, bool have_aux) {
  const int64_t w0 = (stride + 31) / 32, w1 = ((stride + 7) / 8 + 31) / 32;
  size_t b = (static_cast<size_t>(rows) * (w0 + w1) * 4 + 255) & ~size_t(255);
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
  uint32_t *bitmap = reinterpret_cast<uint32_t *>(w);
  const int64_t w0 = (a.stride + 31) / 32, w1 = ((a.stride + 7) / 8 + 31) / 32;
  const size_t off = (static_cast<size_t>(a.rows) * (w0 + w1) * 4 + 255) & ~size_t(255);
  const int64_t aux_row = aux_row_bytes(a.stride);
  const uint8_t *aux = a.aux;
  if (!aux) {
    uint8_t *own = w + off;
    cudaError_t e = launch_fill_aux(a, own, s);
    if (e != cudaSuccess) return e;
    aux = own;
  }
  const int nprob = (!a.pool && a.out_pool_blocks > 0) ? 2 : 1;
  const int64_t max_slots = a.pool ? static_cast<int64_t>(a.pool_blocks) * a.bs : a.stride;
  if (max_slots <= kRowMaxSlots && static_cast<int64_t>(a.rows) * nprob * 4 > 2 * device_sm_count()) {
    // more (row, problem) clusters of four than one wave of two CTAs per SM
    // holds: one CTA per (row, problem) instead
    const int smem = static_cast<int>(sizeof(RowSmem));
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(k_select_row), smem);
    if (e != cudaSuccess) return e;
    k_select_row<<<dim3(a.rows, nprob), kRowThreads, smem, s>>>(a, aux, aux_row);
    return cudaGetLastError();
  }
  // CTAs per (row, problem): 8 for long rows while the launch still fits one wave
  // of two CTAs per SM, else 4
  const int ncl = (a.rows * nprob * kSelClusterMax <= 2 * device_sm_count() && w0 >= 4096) ? kSelClusterMax : 4;
  const int64_t slice = span_words(w0, ncl);
  const int in_smem = slice <= kSmemBitmapWords ? 1 : 0;
  const int smem = static_cast<int>(sizeof(SelSmem) + (in_smem ? slice * 4 : 0));
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(k_select), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncl, a.rows, nprob);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute cl[1];
  cl[0].id = cudaLaunchAttributeClusterDimension;
  cl[0].val.clusterDim.x = ncl;
  cl[0].val.clusterDim.y = 1;
  cl[0].val.clusterDim.z = 1;
  cfg.attrs = cl;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_select, a, aux, aux_row, bitmap, in_smem, ncl);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace csa2
