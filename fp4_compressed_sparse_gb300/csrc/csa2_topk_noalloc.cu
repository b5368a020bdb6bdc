// csa2_topk_noalloc.cu -- csa2_topk for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or anything that allocates)
// once they are running: a host framework that owns every device allocation and
// hands plugins only the tensors it created, a real-time service whose memory
// budget is fixed at start-up, or code that must not trigger the allocator's
// implicit device synchronisation.  csa2_topk needs a caller workspace for its
// score histograms, selection state and candidate lists; this variant keeps
// that scratch in a fixed array compiled into the library instead, so the
// caller passes only its inputs and outputs (and no score sideband: it is
// always rebuilt from the scores, inside the array).
//
// The array (kNoAllocScratchBytes, 4 MiB) lives in every GPU that loads the
// library until the process exits.  All calls share it: two calls whose kernels
// overlap on the GPU (different streams, no ordering between them) race on it.
// The histograms are cleared at the start of every call and the selection
// state is written before it is read; nothing in the array needs a known value
// on entry.
//
// Host code must not hand g_topk_scratch itself to a kernel: on the host that
// name is a stand-in, not a device address.  The first call on each device,
// with that device current, asks the runtime for the array's device address
// (cudaGetSymbolAddress) and keeps it for the rest of the process; the address
// belongs to the device's current context, so a cudaDeviceReset after that
// first call is not supported.
#include <cstdio>
#include <mutex>

#include "csa2_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_topk_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_topk_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" csa2_status csa2_topk_noalloc(const float *scores, int64_t score_stride, int32_t batch, int32_t ratio,
                                         const int64_t *q_pos, const int32_t *pool, int32_t pool_blocks,
                                         int32_t pool_block_size, int32_t k, int32_t *idx_out,
                                         int32_t out_pool_blocks, int32_t *pool_out, int32_t *pool_count,
                                         int32_t *err_word, csa2_stream_t stream) {
  CSA2_REQUIRE_PTR(scores);
  CSA2_REQUIRE_PTR(q_pos);
  CSA2_REQUIRE_PTR(idx_out);
  CSA2_REQUIRE(batch >= 1 && batch <= 65535, CSA2_ERR_SHAPE, "batch %d outside 1..65535", batch);
  CSA2_REQUIRE(score_stride >= 1, CSA2_ERR_SHAPE, "score_stride %lld < 1", static_cast<long long>(score_stride));
  CSA2_REQUIRE(ratio == 1 || ratio == 2, CSA2_ERR_RANGE, "ratio %d (must be 1 or 2)", ratio);
  CSA2_REQUIRE(k >= 1 && k <= CSA2_MAX_TOPK, CSA2_ERR_RANGE, "k %d outside 1..2048", k);
  CSA2_REQUIRE(pool_block_size >= 1 && pool_block_size <= 64, CSA2_ERR_SHAPE, "pool_block_size %d outside 1..64",
               pool_block_size);
  if (pool) {
    CSA2_REQUIRE_PTR(pool);
    CSA2_REQUIRE(pool_blocks >= 1, CSA2_ERR_SHAPE, "pool_blocks %d < 1", pool_blocks);
    CSA2_REQUIRE(score_stride >= static_cast<int64_t>(pool_blocks) * pool_block_size, CSA2_ERR_SHAPE,
                 "score_stride %lld < pool_blocks*pool_block_size", static_cast<long long>(score_stride));
    CSA2_REQUIRE(pool_out == nullptr, CSA2_ERR_RANGE, "a pool can only be built in FULL mode");
  }
  if (pool_out) {
    CSA2_REQUIRE_PTR(pool_out);
    CSA2_REQUIRE_PTR(pool_count);
    CSA2_REQUIRE(out_pool_blocks >= 1 && out_pool_blocks <= CSA2_MAX_TOPK, CSA2_ERR_RANGE,
                 "out_pool_blocks %d outside 1..2048", out_pool_blocks);
    CSA2_REQUIRE(pool_block_size == 8, CSA2_ERR_UNSUPPORTED, "the candidate pool is built from 8-position blocks");
  }
  // the same scratch layout csa2_topk uses for its caller workspace
  const size_t need = csa2::topk_workspace_bytes(batch, score_stride, false);
  CSA2_REQUIRE(need <= kNoAllocScratchBytes, CSA2_ERR_WORKSPACE,
               "csa2_topk_noalloc: batch %d x score_stride %lld needs %zu bytes of scratch; the built-in array "
               "holds %zu (use csa2_topk with a caller workspace)",
               batch, static_cast<long long>(score_stride), need, kNoAllocScratchBytes);
  void *ws = nullptr;
  const csa2_status st = csa2::cuda_status(scratch_address(&ws), "csa2_topk_noalloc scratch address");
  if (st != CSA2_OK) return st;
  csa2::TopkArgs a{};
  a.rows = batch;
  a.scores = scores;
  a.stride = score_stride;
  a.aux = nullptr;
  a.ratio = ratio;
  a.q_pos = q_pos;
  a.pool = pool;
  a.pool_blocks = pool_blocks;
  a.bs = pool_block_size;
  a.k = k;
  a.idx_out = idx_out;
  a.out_pool_blocks = pool_out ? out_pool_blocks : 0;
  a.pool_out = pool_out;
  a.pool_count = pool_count;
  a.err = err_word;
  return csa2::cuda_status(csa2::launch_topk(a, ws, reinterpret_cast<cudaStream_t>(stream)),
                           "csa2_topk_noalloc launch");
}
