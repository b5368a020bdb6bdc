// csa2_score_tc.cu -- lightning-indexer scores on the 5th-generation tensor cores.
//
// [P5] "DeepSeek-V4: Towards Highly Efficient Million-Token Context
// Intelligence" §2.3.1: I_{t,s} = sum_h w_{t,h} * ReLU(q_{t,h} . K_s); §2.3.4:
// the indexer QK product runs in FP4.  Keys and queries are MXFP4 (E2M1 with an
// E8M0 scale per 32), which is exactly the operand format of
// tcgen05.mma kind::mxf4 block_scale: the tensor core applies both scales and
// accumulates in fp32.  Each 32-wide block sum of E2M1 products is an exact
// small integer, so every accumulator holds the fp32 value of the exact dot
// whenever that value is representable (block exponents of a pair within 9
// binades) -- the same number the CUDA-core path and the oracle produce.
//
// One 128-key tile = one MMA pair: M = 128 keys (TMEM lanes), N = padded
// indexer heads (TMEM columns), K = 128 (two K=64 instructions).  The epilogue
// thread of a key reads its N accumulators and runs the fixed-order chain
// acc = fma(w_h, max(d_h, +0), acc).
//
// Exactness: a block sum is an integer below 2^13, and with 4 blocks the dot is
// an integer multiple of its smallest block's unit below 2^(15 + span), where
// span = max - min of the pair's block exponents e_q,j + e_k,j.  With span <= 9
// it fits the 24-bit fp32 significand, so the tensor core's fp32 result is the
// exact dot, rounded once (the value the oracle defines).  The epilogue checks
// every visible key against that bound (blocks whose scale code is 0 -- all-zero
// blocks -- take no part) and raises CSA2_DEVERR_INEXACT if some (head, key)
// pair exceeds it: the key's own code spread plus the row's widest query spread
// bounds all its pairs, and only when that sum exceeds 9 is each head checked.
//
// Persistent CTA per SM, warp-specialised (tile j of a CTA, counted over the
// tiles of its item range, goes to producer j % 2, issuer j % 2 and
// accumulator j % kAcc):
//   warps 0, 1  producers (a single thread issuing every bulk copy caps the
//               stream well below HBM speed).  FULL: lane 0 of each warp issues
//               two bulk copies per tile (8 KB codes + 512 B scales, already
//               stored in the MMA operand layout) into a 14-stage ring.  POOL
//               (Reindex): all 32 lanes of both warps gather the tile's 16 pool
//               blocks with zero-filling cp.async, four tiles in flight per warp.
//               Warp 0 also loads each row's query record into one of two B
//               slots.
//   warps 2, 3  MMA issuers (one thread each): scale factors to TMEM
//               (tcgen05.cp), the two MMAs, commits that release the stage and
//               hand the accumulator over.
//   the rest    epilogue: four warps (one per 32-lane TMEM quarter) per
//               accumulator, six accumulators (four or two when 6 x N columns
//               do not fit TMEM beside the scale factors).  A thread owns one key: it
//               reads the key's N accumulator columns and runs the fixed-order
//               chain.  With a sideband buffer the epilogue also histograms the
//               score keys (and, in FULL mode, the 8-position block maxima) in
//               shared memory and adds them to the row's global histogram once
//               the CTA is done with the row, so top-k needs no pass of its own.
//               Each epilogue thread also reads its key's four block scale
//               codes from the scale-factor columns the MMA used (TMEM) and
//               checks the exactness bound for its key.
// Every mbarrier wait is bounded; a wait that runs out raises
// CSA2_DEVERR_TIMEOUT, sets a CTA abort flag and the CTA drains and exits.
#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {
namespace {

// Every role that waits on an mbarrier waits on each of its phases in order:
// a parity wait on a barrier two phases behind the waiter would return at
// once.  So tile j goes to producer j % 2, to MMA issuer j % 2 and to
// accumulator j % kAcc with kAcc a multiple of 2 (issuer i alone feeds the
// accumulators i, i + 2, ...), and the stage count is even: each role then owns
// a fixed subset of the stages and of the accumulators and visits their phases
// consecutively.
constexpr int kProducers = 2;            // copy-issuing warps (FULL mode), alternate tiles
constexpr int kIssuers = 2;              // MMA-issuing warps, alternate tiles
constexpr int kStages = 14;
// TMEM accumulator buffers (tiles in flight in the epilogue): four while they
// and the scale-factor columns fit the 512 TMEM columns, else two
__host__ __device__ constexpr int acc_of(int np) {
  return 6 * np + 8 * 6 + 8 * 2 * kIssuers <= 512 ? 6 : 4 * np + 8 * 4 + 8 * 2 * kIssuers <= 512 ? 4 : 2;
}
constexpr int kAccMax = 6;
static_assert(kStages % kProducers == 0 && kStages % kIssuers == 0, "each role must own whole stages");
constexpr int kFirstEpiWarp = kProducers + kIssuers;
// four epilogue warps (one per TMEM lane quarter) per accumulator
__host__ __device__ constexpr int threads_of(int np) { return 32 * (kFirstEpiWarp + 4 * acc_of(np)); }
constexpr int kStageBytes = kIdxTileCodeBytes + kIdxTileScaleBytes;  // 8704
constexpr int kMaxRowsPerCta = 256;
constexpr int kGatherDepth = 4;          // POOL: gathered tiles in flight per producer warp
constexpr int kTouchCap = 2048;          // touched bins listed per histogram (more: the flush scans them all)
constexpr int kRound = 16;               // accumulator columns read per TMEM load round in the epilogue
constexpr uint32_t kWaitIters = 200;  // suspended polls of <= 1 ms each: a wait gives up after ~0.2 s

// Per-row query record built by k_qprep: B codes (NP x 64 B, K-major no-swizzle:
// chunk c of head h at c*NP*16 + h*16), SFB atom (512 B), w (NP floats).
__host__ __device__ __forceinline__ int qrec_bytes(int np) { return np * 64 + 512 + np * 4; }

// grid (rows, np / 8), 256 threads: one warp per (row, head); lane l quantises
// dims 4l..4l+3 (MX block l / 8; the block's amax is a max over its 8 lanes).
// With a sideband the blocks of a row also clear its two histograms, which
// the score kernel then accumulates.
__global__ void __launch_bounds__(256) k_qprep(const uint16_t *q_idx, const float *w, int H, int np, uint8_t *out,
                                               uint8_t *aux, int64_t aux_row) {
  const int r = blockIdx.x, lane = threadIdx.x & 31;
  // the scan may start its prologue and key-tile copies now; it waits for this
  // grid before it reads a query record or adds to a histogram
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  if (aux) {
    uint4 *hz = reinterpret_cast<uint4 *>(aux + static_cast<size_t>(r) * aux_row);
    constexpr int kVec = 2 * kSelBins * 4 / 16;
    for (int i = blockIdx.y * 256 + threadIdx.x; i < kVec; i += gridDim.y * 256) hz[i] = make_uint4(0, 0, 0, 0);
  }
  const int h = blockIdx.y * 8 + (threadIdx.x >> 5);
  uint8_t *rec = out + static_cast<size_t>(r) * qrec_bytes(np);
  uint8_t *sfb = rec + np * 64;
  if (blockIdx.y == 0) {
    // scale-factor rows of heads np..127 are never written below: zero them
    for (int i = threadIdx.x; i < 512; i += blockDim.x)
      if ((i / 16) + 32 * ((i % 16) / 4) >= np) sfb[i] = 0;
    float *wr = reinterpret_cast<float *>(sfb + 512);
    for (int j = threadIdx.x; j < np; j += blockDim.x) wr[j] = j < H ? w[static_cast<size_t>(r) * H + j] : 0.0f;
  }
  if (h >= np) return;
  float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (h < H) {
    const uint2 u = *reinterpret_cast<const uint2 *>(q_idx + (static_cast<size_t>(r) * H + h) * kDi + 4 * lane);
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xFFFF0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xFFFF0000u);
  }
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  uint32_t codes = 0, sc = 0;
  if (amax != 0.0f) {
    // MXFP4: e = floor(log2 amax) - 2 (clamped to [-127, 127]); codes E2M1(x * 2^-e)
    int e = floor_log2f(amax) - 2;
    e = max(-127, min(127, e));
    const float inv = pow2f(-e);
#pragma unroll
    for (int i = 0; i < 4; ++i) codes |= e2m1_code(__fmul_rn(x[i], inv)) << (4 * i);
    sc = static_cast<uint32_t>(e + 127);
  }
  const int blk = lane >> 3;
  *reinterpret_cast<uint16_t *>(rec + blk * np * 16 + h * 16 + 2 * (lane & 7)) = static_cast<uint16_t>(codes);
  if ((lane & 7) == 0) sfb[16 * (h % 32) + 4 * (h / 32) + blk] = static_cast<uint8_t>(sc);
}

struct TcArgs {
  ScoreArgs s;
  const uint8_t *qrec;  // [rows][qrec_bytes(np)]
  int np;               // heads padded to a multiple of 16
  int ncols;            // TMEM columns allocated
};

__device__ __forceinline__ int64_t row_slots(const TcArgs &a, int r) {
  if (a.s.pool) return static_cast<int64_t>(a.s.pool_blocks) * a.s.pool_bs;
  int64_t T = a.s.q_pos[r] / a.s.ratio;
  if (T < 0) T = 0;
  return min(T, min(a.s.cap, a.s.stride));
}
__device__ __forceinline__ int row_tiles(const TcArgs &a, int r) {
  return static_cast<int>((row_slots(a, r) + kIdxTile - 1) / kIdxTile);
}

struct __align__(1024) Smem {
  uint8_t stage[kStages][kStageBytes];
  uint8_t bslot[2][128 * 64 + 512 + 128 * 4];
  // mbarriers in their own 128-byte lines: generic loads/stores that share a
  // line with them slow every barrier operation down
  __align__(128) uint64_t full[kStages];
  __align__(128) uint64_t empty[kStages];
  __align__(128) uint64_t tfull[kAccMax];
  __align__(128) uint64_t tempty[kAccMax];
  __align__(128) uint64_t bfull[2];
  __align__(128) uint64_t bempty[2];
  __align__(128) uint32_t tmem;
  int abort;   // written only when a wait gives up
  int issued[kProducers];  // tiles whose copies each producer started (written once, at exit)
  __align__(128) int nt[kMaxRowsPerCta];  // visible tiles of the rows this CTA touches (row - row0)
  uint32_t hist[2][kSelBins];  // this CTA's share of the current row's sideband histograms
  uint16_t touched[2][kTouchCap];  // the bins of hist[h] that went from 0 to 1 in the current row
  int ntouched[2];
};
static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "score kernel shared memory above the per-CTA limit");

// Bounded wait for one thread; a wait that runs out raises the timeout bit.
__device__ __forceinline__ bool wait1(Smem &sm, uint64_t *bar, uint32_t phase, int32_t *err) {
  if (tc::mbar_wait_bounded(bar, phase, kWaitIters)) return true;
  *reinterpret_cast<volatile int *>(&sm.abort) = 1;
  raise_err(err, CSA2_DEVERR_TIMEOUT);
  return false;
}

// Warp-uniform bounded wait: lane 0 waits, the whole warp gets the same answer.
__device__ __forceinline__ bool wait_warp(Smem &sm, uint64_t *bar, uint32_t phase, int32_t *err) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait1(sm, bar, phase, err) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Bounded wait by lane 0 for the whole warp; once it succeeds every lane
// observes the completed phase itself (its acquire of the copied data).  The
// phase cannot move on meanwhile: the waiter has not released the buffer yet.
__device__ __forceinline__ bool wait_all(Smem &sm, uint64_t *bar, uint32_t phase, int32_t *err) {
  if (!wait_warp(sm, bar, phase, err)) return false;
  tc::mbar_wait_bounded(bar, phase, kWaitIters);
  return true;
}

// Exactness bound of the block-scaled dot (see the file header).
constexpr int kMaxExactSpan = 9;
// max - min of the nonzero E8M0 codes of the four blocks packed in w (0 if fewer than two)
__device__ __forceinline__ int code_span(uint32_t w) {
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
// span of the exponents e_q,j + e_k,j over the blocks where both codes are nonzero
__device__ __forceinline__ int pair_span(uint32_t wq, uint32_t wk) {
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
// the four block scale codes of query head h in a record's scale-factor atom
__device__ __forceinline__ uint32_t sfb_word(const uint8_t *sf, int h) {
  return *reinterpret_cast<const uint32_t *>(sf + 16 * (h % 32) + 4 * (h / 32));
}

__device__ __forceinline__ uint32_t sel_key(float f) { return isnan(f) ? 0u : orderable(f); }

// Count one key in bin b of histogram h; a bin's first key also lists the bin.
// atomic add on a shared-memory word, returning the old value (shared-space
// atomics: the Smem reference alone does not tell the compiler the space)
__device__ __forceinline__ uint32_t atom_add_shared(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared.add.u32 %0, [%1], %2;\n" : "=r"(old) : "r"(tc::smem_addr(p)), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void note_bin(Smem &sm, int h, uint32_t b) {
  if (atom_add_shared(&sm.hist[h][b], 1u) == 0u) {
    const int k = static_cast<int>(atom_add_shared(reinterpret_cast<uint32_t *>(&sm.ntouched[h]), 1u));
    if (k < kTouchCap) sm.touched[h][k] = static_cast<uint16_t>(b);
  }
}

// Named barrier over `count` threads returning the AND of `v` across them.
__device__ __forceinline__ int bar_and(uint32_t id, uint32_t count, int v) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.s32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v), "r"(id), "r"(count)
      : "memory");
  return r;
}
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// the same with an L2 cache policy (createpolicy)
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(tc::smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(tc::smem_addr(bar))
               : "memory");
}

// kFullAux: the Full-layer scan with a sideband (no pool, aux present), fixed at
// compile time so that its per-key path carries no mode tests
// Modes fixed at compile time, so that the per-key path carries no mode tests:
//   kModeGeneric   FULL or POOL, with or without a sideband
//   kModeFullAux   FULL with the whole sideband (score histogram, 8-position
//                  block maxima and their histogram: top-k can build a pool)
//   kModeFullHist  FULL with the score histogram alone (the chunked prefill,
//                  whose top-k builds no pool)
constexpr int kModeGeneric = 0, kModeFullAux = 1, kModeFullHist = 2;

template <int NP, int kMode>
__global__ void __launch_bounds__(threads_of(NP), 1) k_index_score_tc(TcArgs a, int max_tiles, int64_t total_items,
                                                                int64_t per_cta) {
  constexpr bool kFullAux = kMode == kModeFullAux, kFullHist = kMode == kModeFullHist;
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * per_cta;
  const int64_t i1 = min(total_items, i0 + per_cta);
  // items are (row, tile < max_tiles), row-major; a tile past the row's visible
  // length is empty and every role skips it the same way
  constexpr int np = NP;
  constexpr int kAcc = acc_of(NP), kEpiWarps = 4 * kAcc;
  static_assert(kAcc % kIssuers == 0, "each accumulator must be fed by one issuer");
  const int brec = qrec_bytes(np);
  const bool pool_mode = (kFullAux || kFullHist) ? false : a.s.pool != nullptr;
  const bool has_aux = (kFullAux || kFullHist) ? true : a.s.aux != nullptr;
  const int64_t seq_tiles = idx_tiles(a.s.cap);

  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem, a.ncols);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&sm.full[s], 1);
      tc::mbar_init(&sm.empty[s], 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      tc::mbar_init(&sm.tfull[i], 1);
      tc::mbar_init(&sm.tempty[i], 4);  // the four warps of the accumulator's epilogue group
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm.bfull[i], 1);
      tc::mbar_init(&sm.bempty[i], kIssuers + kEpiWarps);
    }
    sm.abort = 0;
    sm.ntouched[0] = sm.ntouched[1] = 0;
    for (int i = 0; i < kProducers; ++i) sm.issued[i] = 0;
    tc::fence_mbar_init();
  }
  // visible tile count of every row in this CTA's item range, computed once
  const int row0 = static_cast<int>(i0 / max_tiles);
  const int row_last = i1 > i0 ? static_cast<int>((i1 - 1) / max_tiles) : row0;
  const int nrows = row_last - row0 + 1;
  for (int r = threadIdx.x; r < nrows && r < kMaxRowsPerCta; r += blockDim.x) sm.nt[r] = row_tiles(a, row0 + r);
  for (int i = threadIdx.x; i < 2 * kSelBins; i += blockDim.x) (&sm.hist[0][0])[i] = 0;
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem;
  auto tiles_of = [&](int row) -> int {
    const int k = row - row0;
    return k < kMaxRowsPerCta ? sm.nt[k] : row_tiles(a, row);
  };
  // TMEM columns: accumulators [0, kAcc*np), SFA per accumulator at kAcc*np + 8*i,
  // SFB per B slot at kAcc*np + 8*kAcc + 8*i
  // SFB: one copy per (issuer, B slot) at col_sfb + 8 * (2 * issuer + slot)
  const uint32_t col_sfa = kAcc * np, col_sfb = kAcc * np + 8 * kAcc;

  // Every role walks the rows of the CTA's item range in order and, in each
  // row with visible tiles, visits its own tiles directly: tile j (counted over
  // the visible tiles of the range) belongs to producer j % 2, issuer j % 2 and
  // accumulator j % kAcc.
  const int tile_begin = static_cast<int>(i0 - static_cast<int64_t>(row0) * max_tiles);
  // visible tiles [t0, t1) of row r inside the item range
  auto row_span = [&](int r, int &t0, int &t1) {
    t0 = r == row0 ? tile_begin : 0;
    const int end_item = r == row_last ? static_cast<int>(i1 - static_cast<int64_t>(row_last) * max_tiles) : max_tiles;
    t1 = min(end_item, tiles_of(r));
  };
  // the first tile t >= t0 of a row whose visible tiles start at count jrow with (jrow + t - t0) % mod == q
  auto first_own = [](int t0, int jrow, int mod, int q) { return t0 + ((q - jrow % mod) % mod + mod) % mod; };

  if (warp < kProducers && (lane == 0 || pool_mode)) {
    // ------------------------------------------------------------ producers
    // FULL: lane 0 of each producer warp, alternate tiles, two bulk copies per
    // tile.  POOL: every lane of each producer warp, alternate tiles, gathering
    // with cp.async; a warp keeps kGatherDepth tiles in flight and hands a tile
    // over once its copies have landed.  Producer 0 also loads each row's query
    // record into a B slot.
    const int pw = warp, nprod = kProducers;
    const uint64_t pol = policy_evict_first();  // each key tile is read once per call
    int bchanges = 0, jrow = 0, mine = 0;
    bool ok = true;
    int npend = 0, jlast = 0;  // POOL: own tiles in flight, the newest one's index
    auto hand_over = [&](int st) {
      tc::fence_proxy_async_smem();  // the gathered tile is read by the tensor cores
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.full[st]);
    };
    for (int row = row0; row <= row_last && ok; ++row) {
      int t0, t1;
      row_span(row, t0, t1);
      if (t1 <= t0) continue;
      const int bs = bchanges & 1;
      if (pw == 0) {
        if (bchanges == 0) asm volatile("griddepcontrol.wait;\n" ::: "memory");  // the query prep is complete
        if (bchanges >= 2) {
          if (pool_mode) {
            // the slot is freed by the MMAs of two rows back, which may need tiles
            // this warp still has in flight: hand every one of them over first
            asm volatile("cp.async.wait_group 0;\n" ::: "memory");
            for (; npend > 0; --npend) hand_over((jlast - (npend - 1) * nprod) % kStages);
          }
          ok = pool_mode ? wait_warp(sm, &sm.bempty[bs], ((bchanges >> 1) - 1) & 1, a.s.err)
                         : wait1(sm, &sm.bempty[bs], ((bchanges >> 1) - 1) & 1, a.s.err);
          if (!ok) break;
        }
        if (lane == 0) {
          tc::mbar_expect_tx(&sm.bfull[bs], brec);
          bulk_g2s(tc::smem_addr(sm.bslot[bs]), a.qrec + static_cast<size_t>(row) * brec, brec, &sm.bfull[bs]);
        }
      }
      ++bchanges;
      const int seq = a.s.cache_seq < 0 ? row : a.s.cache_seq;
      // FULL: the physical tile of the next own tile is looked up one step ahead,
      // so that a paged cache's table read overlaps the wait for a free stage
      const int tile_first = first_own(t0, jrow, nprod, pw);
      int64_t t_next = (!pool_mode && tile_first < t1) ? phys_tile(a.s.map, seq, tile_first) : 0;
      for (int tile = tile_first; tile < t1; tile += nprod) {
        const int j = jrow + (tile - t0), s = j % kStages;
        const int64_t t = t_next;
        if (!pool_mode && tile + nprod < t1) t_next = phys_tile(a.s.map, seq, tile + nprod);
        if (j >= kStages) ok = pool_mode ? wait_warp(sm, &sm.empty[s], ((j / kStages) - 1) & 1, a.s.err)
                                         : wait1(sm, &sm.empty[s], ((j / kStages) - 1) & 1, a.s.err);
        if (!ok) break;
        uint8_t *dst = sm.stage[s];
        if (!pool_mode) {
          if (t >= 0) {
            tc::mbar_expect_tx(&sm.full[s], kStageBytes);
            bulk_g2s_hint(tc::smem_addr(dst), a.s.idx_codes + static_cast<size_t>(t) * kIdxTileCodeBytes,
                          kIdxTileCodeBytes, &sm.full[s], pol);
            bulk_g2s_hint(tc::smem_addr(dst + kIdxTileCodeBytes),
                          a.s.idx_scales + static_cast<size_t>(t) * kIdxTileScaleBytes, kIdxTileScaleBytes, &sm.full[s],
                          pol);
          } else {  // a page id outside the pool: the tile is not read (its scores are unspecified)
            raise_err(a.s.err, CSA2_DEVERR_INDEX);
            tc::mbar_arrive(&sm.full[s]);
          }
        } else {
          // 16 pool blocks of 8 keys: lane l gathers block l/2, code chunks 2*(l%2)..+1
          // and 4 of its scale words; outside the pool or the cache the copy reads
          // nothing and writes zeros
          const int jb = lane >> 1;
          const int pidx = tile * 16 + jb;
          const int32_t pid =
              pidx < a.s.pool_blocks ? a.s.pool[static_cast<size_t>(row) * a.s.pool_blocks + pidx] : -1;
          const int64_t p0 = static_cast<int64_t>(pid) * a.s.pool_bs;
          const int64_t pt = (pid >= 0 && p0 + a.s.pool_bs <= seq_tiles * kIdxTile) ? phys_tile(a.s.map, seq, p0 / kIdxTile)
                                                                                   : -1;
          const bool okb = pt >= 0;
          const uint32_t d0 = tc::smem_addr(dst);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * (lane & 1) + cc;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint8_t *src = okb ? a.s.idx_codes + idx_code_at(pt, static_cast<int>((p0 + i) % kIdxTile), c)
                                       : a.s.idx_codes;
              asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d0 + c * 2048 + (jb * 8 + i) * 16),
                           "l"(src), "r"(okb ? 16 : 0)
                           : "memory");
            }
          }
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            const int i = (lane & 1) * 4 + i4, m = jb * 8 + i;
            const uint8_t *src = okb ? a.s.idx_scales + idx_scale_at(pt, static_cast<int>((p0 + i) % kIdxTile))
                                     : a.s.idx_scales;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(
                             d0 + kIdxTileCodeBytes + 16 * (m % 32) + 4 * (m / 32)),
                         "l"(src), "r"(okb ? 4 : 0)
                         : "memory");
          }
          asm volatile("cp.async.commit_group;\n" ::: "memory");
          jlast = j;
          if (++npend == kGatherDepth) {
            // the oldest tile in flight has landed: hand it over
            asm volatile("cp.async.wait_group %0;\n" ::"n"(kGatherDepth - 1) : "memory");
            hand_over((jlast - (npend - 1) * nprod) % kStages);
            --npend;
          }
        }
        mine = j + 1;
      }
      jrow += t1 - t0;
    }
    if (pool_mode) {  // every gathered tile still in flight (also after a wait gave up)
      asm volatile("cp.async.wait_group 0;\n" ::: "memory");
      for (; npend > 0; --npend) hand_over((jlast - (npend - 1) * nprod) % kStages);
    }
    if (lane == 0) sm.issued[pw] = mine;
  } else if (warp >= kProducers && warp < kProducers + kIssuers && lane == 0) {
    // ------------------------------------------------------------ MMA issuers (one thread each)
    // issuer `who` takes the CTA's tiles j with j % kIssuers == who (accumulators
    // and stages who, who + kIssuers, ...); each keeps its own copy of the row's
    // query scale factors in TMEM
    const int who = warp - kProducers;
    int bchanges = 0, jrow = 0;
    const uint32_t id0 = tc::idesc_mxf4(128, np, 0, 0), id1 = tc::idesc_mxf4(128, np, 2, 2);
    bool dead = false;
    for (int row = row0; row <= row_last && !dead; ++row) {
      int t0, t1;
      row_span(row, t0, t1);
      if (t1 <= t0) continue;
      const int bs = bchanges & 1;
      if (!wait1(sm, &sm.bfull[bs], (bchanges >> 1) & 1, a.s.err)) {
        dead = true;
        break;
      }
      ++bchanges;
      tc::tc_fence_after();
      const uint32_t sfb = tmem + col_sfb + 8 * (2 * who + bs);
      tc::tmem_cp_32x128b_x4(sfb, tc::smem_desc_noswizzle(tc::smem_addr(sm.bslot[bs] + np * 64), 128, 128));
      for (int tile = first_own(t0, jrow, kIssuers, who); tile < t1; tile += kIssuers) {
        const int j = jrow + (tile - t0), s = j % kStages, acc = j % kAcc;
        if (!wait1(sm, &sm.full[s], (j / kStages) & 1, a.s.err) ||
            (j >= kAcc && !wait1(sm, &sm.tempty[acc], ((j / kAcc) - 1) & 1, a.s.err))) {
          dead = true;
          break;
        }
        tc::tc_fence_after();
        const uint32_t sa = tc::smem_addr(sm.stage[s]), sb = tc::smem_addr(sm.bslot[bs]);
        tc::tmem_cp_32x128b_x4(tmem + col_sfa + 8 * acc, tc::smem_desc_noswizzle(sa + kIdxTileCodeBytes, 128, 128));
        const uint32_t d = tmem + acc * np;
        tc::mma_mxf4(d, tc::smem_desc_noswizzle(sa, 2048, 128), tc::smem_desc_noswizzle(sb, np * 16, 128), id0,
                     tmem + col_sfa + 8 * acc, sfb, 0);
        tc::mma_mxf4(d, tc::smem_desc_noswizzle(sa + 4096, 2048, 128),
                     tc::smem_desc_noswizzle(sb + 2 * np * 16, np * 16, 128), id1, tmem + col_sfa + 8 * acc, sfb, 1);
        tc::mma_commit(&sm.empty[s]);
        tc::mma_commit(&sm.tfull[acc]);
      }
      // the row's B slot is free once both issuers' MMAs of the row are done
      if (!dead) tc::mma_commit(&sm.bempty[bs]);
      jrow += t1 - t0;
    }
  } else if (warp >= kFirstEpiWarp) {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kFirstEpiWarp;  // 0 .. kEpiWarps-1
    const int parity = e >> 2;        // accumulator buffer this warp drains (tiles j % kAcc == parity)
    const int quarter = warp & 3;     // TMEM lane quarter this warp may access
    const int m = 32 * quarter + lane;
    const int64_t aux_row = aux_row_bytes(a.s.stride);
    int bchanges = 0, jrow = 0;
    bool dead = false;
    for (int row = row0; row <= row_last; ++row) {
      int t0, t1;
      row_span(row, t0, t1);
      if (t1 <= t0) continue;
      const int bs = bchanges & 1;
      ++bchanges;
      const int64_t row_nslots = row_slots(a, row);
      const int64_t row_T = pool_mode ? a.s.q_pos[row] / a.s.ratio : 0;  // POOL: visible positions
      const uint8_t *qsf = sm.bslot[bs] + np * 64;  // the row's query scale codes
      int qspan = -1;                               // the widest, read once the record has landed
      for (int tile = first_own(t0, jrow, kAcc, parity); tile < t1 && !dead; tile += kAcc) {
        const int j = jrow + (tile - t0);
        const int64_t slot = static_cast<int64_t>(tile) * kIdxTile + m;
        // POOL: the key's pool block, requested before the wait for the accumulator
        int32_t pid = -1;
        if (pool_mode && slot < static_cast<int64_t>(a.s.pool_blocks) * a.s.pool_bs)
          pid = __ldg(a.s.pool + static_cast<size_t>(row) * a.s.pool_blocks + slot / a.s.pool_bs);
        // each warp of the group waits for the accumulator itself and hands
        // its lane quarter back on its own (tempty counts four arrivals)
        int ok = 1;
        if (lane == 0)
          ok = wait1(sm, &sm.bfull[bs], ((bchanges - 1) >> 1) & 1, a.s.err) &&
               wait1(sm, &sm.tfull[parity], (j / kAcc) & 1, a.s.err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          dead = true;
        } else {
          tc::tc_fence_after();
          if (qspan < 0) {
            qspan = 0;
            for (int h = lane; h < np; h += 32) qspan = max(qspan, code_span(sfb_word(qsf, h)));
            qspan = __reduce_max_sync(0xffffffffu, qspan);
          }
          const float4 *wv = reinterpret_cast<const float4 *>(sm.bslot[bs] + np * 64 + 512);  // head weights
          const uint32_t base = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + parity * np;
          // the key's block scale codes: the scale-factor columns of this accumulator
          // hold, in lane 32q + r, the codes of keys r, r + 32, r + 64, r + 96 (one
          // column each); this thread's key 32 quarter + lane is column `quarter`
          uint32_t kcodes;
          tc::tmem_ld_32x32b_x1(tmem + (static_cast<uint32_t>(32 * quarter) << 16) + col_sfa + 8 * parity + quarter,
                                kcodes);
          // up to kRound columns per round: every load of the round, then one
          // wait; the fma chain runs over the heads in order
          float acc = 0.0f;
#pragma unroll
          for (int h0 = 0; h0 < np; h0 += kRound) {
            constexpr int kMaxC = (np < kRound ? np : kRound) / 16;
            const int nc = (np - h0 < kRound ? np - h0 : kRound) / 16;
            uint32_t r[kMaxC][16];
#pragma unroll
            for (int c = 0; c < kMaxC; ++c)
              if (c < nc) tc::tmem_ld_32x32b_x16(base + h0 + 16 * c, r[c]);
#pragma unroll
            for (int c = 0; c < kMaxC; ++c)
              if (c < nc) tc::tmem_ld_wait_x16(r[c]);
            if (h0 + kRound >= np) {
              // every TMEM read of this warp is complete: hand its quarter back
              tc::tc_fence_before();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sm.tempty[parity]);
            }
#pragma unroll
            for (int c = 0; c < kMaxC; ++c) {
              if (c >= nc) break;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float4 w4 = wv[(h0 + 16 * c) / 4 + q];
                const float wq[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float d = __uint_as_float(r[c][4 * q + k]);
                  acc = __fmaf_rn(wq[k], fmaxf(d, 0.0f), acc);  // ReLU; NaN -> 0, -0 adds nothing
                }
              }
            }
          }
          // kcodes landed with the rounds' waits; keep its uses after them
          asm volatile("" : "+r"(kcodes));
          bool valid;
          if (!pool_mode) {
            valid = slot < row_nslots;
          } else {
            const int64_t p = static_cast<int64_t>(pid) * a.s.pool_bs + slot % a.s.pool_bs;
            valid = pid >= 0 && p < row_T && p < a.s.cap;
            if (pid >= 0 && p >= a.s.cap) raise_err(a.s.err, CSA2_DEVERR_INDEX);
          }
          if (valid) a.s.scores[static_cast<size_t>(row) * a.s.stride + slot] = acc;
          // exactness bound for this key (rarely does it need the per-head check)
          const int kspan = valid ? code_span(kcodes) : 0;
          if (__any_sync(0xffffffffu, kspan + qspan > kMaxExactSpan)) {
            bool bad = false;
            if (kspan + qspan > kMaxExactSpan)
              for (int h = 0; h < np && !bad; ++h) bad = pair_span(sfb_word(qsf, h), kcodes) > kMaxExactSpan;
            if (bad) raise_err(a.s.err, CSA2_DEVERR_INEXACT);
          }
          if (has_aux) {
            // sideband: score-key histogram; FULL rows also the max of each
            // 8-position block (8 consecutive lanes) and its histogram
            if (valid) note_bin(sm, 0, sel_key(acc) >> kSelBinShift);
            if (!pool_mode && !kFullHist) {
              float v = valid ? acc : -INFINITY;
              v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
              v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
              v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
              if ((lane & 7) == 0 && valid) {
                float *bm = reinterpret_cast<float *>(a.s.aux + static_cast<size_t>(row) * aux_row + 2 * kSelBins * 4);
                bm[slot / 8] = v;
                note_bin(sm, 1, sel_key(v) >> kSelBinShift);
              }
            }
          }
        }
      }
      jrow += t1 - t0;
      if (lane == 0) tc::mbar_arrive(&sm.bempty[bs]);
      if (has_aux) {
        if (bchanges == 1) asm volatile("griddepcontrol.wait;\n" ::: "memory");  // the histograms are cleared
        // every epilogue warp is done with this row: add the CTA's histograms
        // to the row's sideband and clear them (only the listed bins, unless
        // more bins were touched than the list holds)
        const int et = threadIdx.x - 32 * kFirstEpiWarp;
        asm volatile("bar.sync 1, %0;\n" ::"r"(kEpiWarps * 32) : "memory");
        const int n0 = sm.ntouched[0], n1 = sm.ntouched[1];
        asm volatile("bar.sync 1, %0;\n" ::"r"(kEpiWarps * 32) : "memory");
        if (et == 0) sm.ntouched[0] = sm.ntouched[1] = 0;
        uint32_t *gh = reinterpret_cast<uint32_t *>(a.s.aux + static_cast<size_t>(row) * aux_row);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = h == 0 ? n0 : n1;
          if (n <= kTouchCap) {
            for (int i = et; i < n; i += kEpiWarps * 32) {
              const uint32_t b = sm.touched[h][i];
              atomicAdd(&gh[h * kSelBins + b], sm.hist[h][b]);
              sm.hist[h][b] = 0;
            }
          } else {
            for (int b = et; b < kSelBins; b += kEpiWarps * 32) {
              const uint32_t c = sm.hist[h][b];
              if (c) {
                atomicAdd(&gh[h * kSelBins + b], c);
                sm.hist[h][b] = 0;
              }
            }
          }
        }
        asm volatile("bar.sync 1, %0;\n" ::"r"(kEpiWarps * 32) : "memory");
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    // copies still in flight (only after an abort): bounded wait on the last items issued
    if (*reinterpret_cast<volatile int *>(&sm.abort) && lane == 0) {  // after a timeout only
      int n = 0;
      for (int i = 0; i < kProducers; ++i) n = max(n, sm.issued[i]);
      for (int jj = n > kStages ? n - kStages : 0; jj < n; ++jj)
        tc::mbar_wait_bounded(&sm.full[jj % kStages], (jj / kStages) & 1, kWaitIters);
    }
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, a.ncols);
  }
}

}  // namespace

size_t score_tc_workspace_bytes(int rows, int heads) {
  const int np = ((heads + 15) / 16) * 16;
  return static_cast<size_t>(rows) * qrec_bytes(np) + 256;
}

cudaError_t launch_index_score_tc(const ScoreArgs &s, void *ws, cudaStream_t st) {
  if (s.rows <= 0) return cudaSuccess;
  TcArgs a{};
  a.s = s;
  a.np = ((s.heads + 15) / 16) * 16;
  a.qrec = static_cast<const uint8_t *>(ws);
  const int cols = acc_of(a.np) * a.np + 8 * acc_of(a.np) + 8 * 2 * kIssuers;
  a.ncols = cols <= 128 ? 128 : (cols <= 256 ? 256 : 512);
  k_qprep<<<dim3(s.rows, a.np / 8), 256, 0, st>>>(s.q_idx, s.w, s.heads, a.np, static_cast<uint8_t *>(ws), s.aux,
                                                  static_cast<int64_t>(aux_row_bytes(s.stride)));
  const int max_tiles = static_cast<int>(
      s.pool ? (static_cast<int64_t>(s.pool_blocks) * s.pool_bs + kIdxTile - 1) / kIdxTile
             : idx_tiles(s.cap < s.stride ? s.cap : s.stride));
  const int64_t total = static_cast<int64_t>(s.rows) * max_tiles;
  if (total <= 0) return cudaGetLastError();
  const int num_sms = device_sm_count();
  const size_t smem = sizeof(Smem) + 1024;
  using KernelFn = void (*)(TcArgs, int, int64_t, int64_t);
  KernelFn fn = nullptr;
  const int mode = (s.pool != nullptr || s.aux == nullptr) ? kModeGeneric : s.no_block_max ? kModeFullHist : kModeFullAux;
#define CSA2_SCORE_FN(N)                                                                  \
  (mode == kModeFullAux ? k_index_score_tc<N, kModeFullAux>                               \
                        : mode == kModeFullHist ? k_index_score_tc<N, kModeFullHist>      \
                                                : k_index_score_tc<N, kModeGeneric>)
  switch (a.np) {
    case 16: fn = CSA2_SCORE_FN(16); break;
    case 32: fn = CSA2_SCORE_FN(32); break;
    case 48: fn = CSA2_SCORE_FN(48); break;
    case 64: fn = CSA2_SCORE_FN(64); break;
    case 80: fn = CSA2_SCORE_FN(80); break;
    case 96: fn = CSA2_SCORE_FN(96); break;
    case 112: fn = CSA2_SCORE_FN(112); break;
    default: fn = CSA2_SCORE_FN(128); break;
  }
#undef CSA2_SCORE_FN
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(fn), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t grid = total < num_sms ? total : num_sms;
  const int64_t per = (total + grid - 1) / grid;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(threads_of(a.np));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlaps the query prep's tail
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a, max_tiles, total, per);
}

}  // namespace csa2
