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
#include <cstdio>
#include <mutex>

#include "csa2_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_topk_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_topk_scratch on the current device (looked up once per
// device; the name alone is a host-side stand-in and must not be passed to a kernel).
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

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" csa2_status csa2_topk_noalloc(const float *scores, int64_t score_stride, int32_t batch, int32_t ratio,
                                         const int64_t *q_pos, const int32_t *pool, int32_t pool_blocks,
                                         int32_t pool_block_size, int32_t k, int32_t *idx_out,
                                         int32_t out_pool_blocks, int32_t *pool_out, int32_t *pool_count,
                                         int32_t *err_word, csa2_stream_t stream) {
  if (!scores || !q_pos || !idx_out) return CSA2_ERR_NULL;
  if (!aligned16(scores) || !aligned16(q_pos) || !aligned16(idx_out)) return CSA2_ERR_ALIGN;
  if (batch < 1 || batch > 65535 || score_stride < 1) return CSA2_ERR_SHAPE;
  if (ratio != 1 && ratio != 2) return CSA2_ERR_RANGE;
  if (k < 1 || k > CSA2_MAX_TOPK) return CSA2_ERR_RANGE;
  if (pool_block_size < 1 || pool_block_size > 64) return CSA2_ERR_SHAPE;
  if (pool) {
    if (!aligned16(pool)) return CSA2_ERR_ALIGN;
    if (pool_blocks < 1 || score_stride < static_cast<int64_t>(pool_blocks) * pool_block_size)
      return CSA2_ERR_SHAPE;
    if (pool_out) return CSA2_ERR_RANGE;
  }
  if (pool_out) {
    if (!pool_count) return CSA2_ERR_NULL;
    if (!aligned16(pool_out) || !aligned16(pool_count)) return CSA2_ERR_ALIGN;
    if (out_pool_blocks < 1 || out_pool_blocks > CSA2_MAX_TOPK) return CSA2_ERR_RANGE;
    if (pool_block_size != 8) return CSA2_ERR_UNSUPPORTED;
  }
  // the same scratch layout csa2_topk uses for its caller workspace
  const size_t need = csa2::topk_workspace_bytes(batch, score_stride, false);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "csa2_topk_noalloc: batch %d x score_stride %lld needs %zu bytes of scratch; the built-in "
             "array holds %zu (use csa2_topk with a caller workspace)",
             batch, static_cast<long long>(score_stride), need, kNoAllocScratchBytes);
    csa2::set_error_detail(msg);
    return CSA2_ERR_WORKSPACE;
  }
  void *ws = nullptr;
  const cudaError_t ce = scratch_address(&ws);
  if (ce != cudaSuccess) {
    csa2::set_error_detail(cudaGetErrorString(ce));
    return CSA2_ERR_CUDA;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
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
  if (csa2::launch_topk(a, ws, s) != cudaSuccess) return CSA2_ERR_CUDA;
  return CSA2_OK;
}
