// csa2_topk.cu -- deterministic top-k selection over index scores, and the
// candidate-pool build of the Hierarchical Sparse Indexer.
//
// [P5] "DeepSeek-V4: Towards Highly Efficient Million-Token Context
// Intelligence" §2.3.1: C^Sprs_t = { C_s | I_{t,s} in Top-k(I_{t,:}) }.
// [P1] "DeepSeek V4.1 Flash 아키텍처 분석" §"512개를 고르기 위해 ...": positions
// grouped 8 at a time, a block ranked by its max score, at most 2,048 blocks kept.
//
// Order: key = orderable(score) (-0 == +0, NaN lowest), descending; ties by the
// lower slot (slots run in ascending position order in every mode).  The k-th
// largest key is found by three histogram passes (11 + 11 + 10 bits) whose
// counts are order-independent; the chosen slots are then compacted in slot
// order with per-CTA counts and prefix sums.  No result depends on scheduling.
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 4096;            // slots per CTA
constexpr int kPerThread = kChunk / kThreads;
constexpr int kBins = 2048;
// radix digits of pass 0, 1, 2: bits 31..21, 20..10, 9..0
__host__ __device__ __forceinline__ int shift_of(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }
__host__ __device__ __forceinline__ uint32_t mask_of(int pass) { return pass < 2 ? 0x7FFu : 0x3FFu; }

struct RowState {
  uint32_t prefix;      // decided high bits of the threshold key
  uint32_t krem;        // how many keys equal to the final threshold to take
  uint32_t total;       // valid slots
  uint32_t select_all;  // total <= k: every valid slot is chosen
};

__device__ __forceinline__ void row_range(const SelArgs &a, int r, int64_t &nslots, int64_t &T) {
  T = a.q_pos[r] / a.ratio;
  if (T < 0) T = 0;
  if (a.mode == kSelPool) {
    // slots are pool positions; the stride bounds the slots, not the positions
    nslots = static_cast<int64_t>(a.pool_blocks) * a.bs;
    return;
  }
  T = min(T, a.stride);  // FULL / BLOCKMAX: slot s is position s
  nslots = a.mode == kSelBlockMax ? (T + a.bs - 1) / a.bs : T;
}

// Key and output position of one slot; false when the slot is not a candidate.
__device__ __forceinline__ bool slot_key(const SelArgs &a, int r, int64_t slot, int64_t T, uint32_t &key,
                                         int32_t &pos) {
  const float *row = a.scores + static_cast<size_t>(r) * a.stride;
  float f;
  if (a.mode == kSelFull) {
    f = row[slot];
    pos = static_cast<int32_t>(slot);
  } else if (a.mode == kSelPool) {
    const int32_t pid = a.pool[static_cast<size_t>(r) * a.pool_blocks + slot / a.bs];
    if (pid < 0) return false;
    const int64_t p = static_cast<int64_t>(pid) * a.bs + slot % a.bs;
    if (p >= T) return false;
    f = row[slot];
    pos = static_cast<int32_t>(p);
  } else {
    const int64_t p0 = slot * a.bs;
    const int64_t p1 = min(p0 + a.bs, T);
    f = -INFINITY;
    for (int64_t p = p0; p < p1; ++p) f = fmaxf(f, row[p]);
    pos = static_cast<int32_t>(slot);
  }
  if (isnan(f)) {
    raise_err(a.err, CSA2_DEVERR_NAN);
    key = 0;
  } else {
    key = orderable(f);
  }
  return true;
}

__device__ __forceinline__ bool key_matches(uint32_t key, int pass, uint32_t prefix) {
  if (pass == 0) return true;
  const int sh = shift_of(pass - 1);
  return (key >> sh) == (prefix >> sh);
}

__global__ void __launch_bounds__(kThreads) k_sel_hist(SelArgs a, int pass, uint32_t *hist,
                                                       const RowState *state) {
  __shared__ uint32_t sh[kBins];
  const int r = blockIdx.y;
  int64_t nslots, T;
  row_range(a, r, nslots, T);
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  if (s0 >= nslots) return;
  RowState st = {0, 0, 0, 0};
  if (pass > 0) {
    st = state[r];
    if (st.select_all) return;
  }
  for (int i = threadIdx.x; i < kBins; i += kThreads) sh[i] = 0;
  __syncthreads();
  const int64_t s1 = min(s0 + kChunk, nslots);
  for (int64_t slot = s0 + threadIdx.x; slot < s1; slot += kThreads) {
    uint32_t key;
    int32_t pos;
    if (slot_key(a, r, slot, T, key, pos) && key_matches(key, pass, st.prefix))
      atomicAdd(&sh[(key >> shift_of(pass)) & mask_of(pass)], 1u);
  }
  __syncthreads();
  uint32_t *g = hist + (static_cast<size_t>(r) * 3 + pass) * kBins;
  for (int i = threadIdx.x; i < kBins; i += kThreads)
    if (sh[i]) atomicAdd(&g[i], sh[i]);
}

// exclusive scan over the block's threads (inclusive result returned in *incl)
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_tot, uint32_t *incl_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  uint32_t before = 0, total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) before += warp_tot[w];
    total += warp_tot[w];
  }
  __syncthreads();
  if (incl_total) *incl_total = total;
  return before + x - v;
}

// One block per row: locate the bin holding the krem-th largest key.
__global__ void __launch_bounds__(kThreads) k_sel_resolve(SelArgs a, int pass, const uint32_t *hist,
                                                          RowState *state) {
  __shared__ uint32_t warp_tot[kThreads / 32];
  const int r = blockIdx.x;
  const uint32_t *g = hist + (static_cast<size_t>(r) * 3 + pass) * kBins;
  RowState st = pass == 0 ? RowState{0, static_cast<uint32_t>(a.k), 0, 0} : state[r];
  if (pass > 0 && st.select_all) return;
  // thread t owns bins counted from the top: bins nb-1-8t .. nb-8-8t (descending)
  const int nb = static_cast<int>(mask_of(pass)) + 1;
  const int per = nb / kThreads;  // 8 or 4
  uint32_t local = 0;
  for (int i = 0; i < per; ++i) local += g[nb - 1 - (threadIdx.x * per + i)];
  uint32_t total;
  uint32_t above = block_excl_scan(local, warp_tot, &total);
  if (pass == 0) {
    st.total = total;
    if (total <= static_cast<uint32_t>(a.k)) {
      if (threadIdx.x == 0) {
        st.select_all = 1;
        state[r] = st;
      }
      return;
    }
  }
  // the crossing bin: above < krem <= above + local
  if (above < st.krem && st.krem <= above + local) {
    uint32_t acc = above;
    for (int i = 0; i < per; ++i) {
      const int bin = nb - 1 - (threadIdx.x * per + i);
      const uint32_t c = g[bin];
      if (acc + c >= st.krem) {
        RowState ns = st;
        ns.prefix = st.prefix | (static_cast<uint32_t>(bin) << shift_of(pass));
        ns.krem = st.krem - acc;
        state[r] = ns;
        break;
      }
      acc += c;
    }
  }
}

__device__ __forceinline__ void classify(const RowState &st, uint32_t key, bool &gt, bool &eq) {
  if (st.select_all) {
    gt = true;
    eq = false;
  } else {
    gt = key > st.prefix;
    eq = key == st.prefix;
  }
}

__global__ void __launch_bounds__(kThreads) k_sel_count(SelArgs a, const RowState *state, uint2 *cnt,
                                                        int nctas) {
  __shared__ uint32_t warp_tot[kThreads / 32];
  const int r = blockIdx.y;
  int64_t nslots, T;
  row_range(a, r, nslots, T);
  const RowState st = state[r];
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  uint32_t ngt = 0, neq = 0;
  for (int i = 0; i < kPerThread; ++i) {
    const int64_t slot = s0 + threadIdx.x * kPerThread + i;
    if (slot >= nslots) break;
    uint32_t key;
    int32_t pos;
    if (!slot_key(a, r, slot, T, key, pos)) continue;
    bool gt, eq;
    classify(st, key, gt, eq);
    ngt += gt;
    neq += eq;
  }
  uint32_t tgt, teq;
  block_excl_scan(ngt, warp_tot, &tgt);
  block_excl_scan(neq, warp_tot, &teq);
  if (threadIdx.x == 0) cnt[static_cast<size_t>(r) * nctas + blockIdx.x] = make_uint2(tgt, teq);
}

__global__ void __launch_bounds__(kThreads) k_sel_write(SelArgs a, const RowState *state, const uint2 *cnt,
                                                        int nctas) {
  __shared__ uint32_t warp_tot[kThreads / 32];
  __shared__ uint32_t s_eqb, s_outb, s_total;
  const int r = blockIdx.y;
  int64_t nslots, T;
  row_range(a, r, nslots, T);
  const RowState st = state[r];
  const uint32_t krem = st.select_all ? 0u : st.krem;
  if (threadIdx.x == 0) {
    // walk the CTAs in slot order: equal keys are taken first-come until krem
    uint32_t eqb = 0, outb = 0, total = 0;
    for (int c = 0; c < nctas; ++c) {
      const uint2 v = cnt[static_cast<size_t>(r) * nctas + c];
      const uint32_t take_eq = min(v.y, krem > eqb ? krem - eqb : 0u);
      if (c == static_cast<int>(blockIdx.x)) {
        s_eqb = eqb;
        s_outb = outb;
      }
      outb += v.x + take_eq;
      eqb += v.y;
    }
    total = outb;
    s_total = total;
  }
  __syncthreads();
  int32_t *out = a.out + static_cast<size_t>(r) * a.out_stride;
  if (blockIdx.x == 0) {
    const uint32_t total = min(s_total, static_cast<uint32_t>(a.k));
    for (int i = static_cast<int>(total) + threadIdx.x; i < a.k; i += kThreads) out[i] = -1;
    if (threadIdx.x == 0 && a.count_out) a.count_out[r] = static_cast<int32_t>(total);
  }
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  if (s0 >= nslots) return;
  // this thread's slots, in order
  uint32_t keys[kPerThread];
  int32_t poss[kPerThread];
  uint8_t flag[kPerThread];  // 1 gt, 2 eq, 0 none
  uint32_t neq = 0;
  for (int i = 0; i < kPerThread; ++i) {
    flag[i] = 0;
    const int64_t slot = s0 + threadIdx.x * kPerThread + i;
    if (slot >= nslots) continue;
    if (!slot_key(a, r, slot, T, keys[i], poss[i])) continue;
    bool gt, eq;
    classify(st, keys[i], gt, eq);
    flag[i] = gt ? 1 : (eq ? 2 : 0);
    neq += eq;
  }
  uint32_t dummy;
  uint32_t eq_before = s_eqb + block_excl_scan(neq, warp_tot, &dummy);
  uint32_t nsel = 0;
  for (int i = 0; i < kPerThread; ++i) {
    if (flag[i] == 2) {
      if (eq_before < krem) flag[i] = 1;
      else flag[i] = 0;
      ++eq_before;
    }
    nsel += flag[i] == 1;
  }
  uint32_t off = s_outb + block_excl_scan(nsel, warp_tot, &dummy);
  for (int i = 0; i < kPerThread; ++i)
    if (flag[i] == 1) {
      if (off < static_cast<uint32_t>(a.k)) out[off] = poss[i];
      ++off;
    }
}

}  // namespace

size_t select_workspace_bytes(int rows, int64_t max_slots) {
  const int64_t nctas = (max_slots + kChunk - 1) / kChunk;
  size_t b = static_cast<size_t>(rows) * 3 * kBins * 4;           // hist
  b += static_cast<size_t>(rows) * sizeof(RowState);              // state
  b = (b + 15) & ~size_t(15);
  b += static_cast<size_t>(rows) * (nctas > 0 ? nctas : 1) * 8;   // counts
  return (b + 255) & ~size_t(255);
}

cudaError_t launch_select(const SelArgs &a, int64_t max_slots, void *ws, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  const int nctas = static_cast<int>(max_slots > 0 ? (max_slots + kChunk - 1) / kChunk : 1);
  uint8_t *p = static_cast<uint8_t *>(ws);
  uint32_t *hist = reinterpret_cast<uint32_t *>(p);
  p += static_cast<size_t>(a.rows) * 3 * kBins * 4;
  RowState *state = reinterpret_cast<RowState *>(p);
  size_t off = static_cast<size_t>(a.rows) * 3 * kBins * 4 + static_cast<size_t>(a.rows) * sizeof(RowState);
  off = (off + 15) & ~size_t(15);
  uint2 *cnt = reinterpret_cast<uint2 *>(static_cast<uint8_t *>(ws) + off);
  cudaError_t e = cudaMemsetAsync(hist, 0, static_cast<size_t>(a.rows) * 3 * kBins * 4, s);
  if (e != cudaSuccess) return e;
  dim3 grid(nctas, a.rows);
  for (int pass = 0; pass < 3; ++pass) {
    k_sel_hist<<<grid, kThreads, 0, s>>>(a, pass, hist, state);
    k_sel_resolve<<<a.rows, kThreads, 0, s>>>(a, pass, hist, state);
  }
  k_sel_count<<<grid, kThreads, 0, s>>>(a, state, cnt, nctas);
  k_sel_write<<<grid, kThreads, 0, s>>>(a, state, cnt, nctas);
  return cudaGetLastError();
}

}  // namespace csa2
