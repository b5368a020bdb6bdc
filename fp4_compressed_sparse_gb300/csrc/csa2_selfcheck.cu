// csa2_selfcheck.cu -- a device self-check of the library's failure path: the
// bounded mbarrier wait every tensor-core kernel uses (producer / issuer /
// epilogue handshakes) gives up after its poll limit, the kernel reports
// CSA2_DEVERR_TIMEOUT in the caller's error word, releases its tensor memory and
// returns, and the context stays usable.  Not a step of the method.
//
// One warp.  Lane 0 initialises an mbarrier expecting one arrival; with
// `complete` set it arrives at once, otherwise nothing ever completes the
// phase.  The warp then holds 32 TMEM columns across a bounded wait of `iters`
// suspended polls (each at most ~1 ms), exactly as the score and attention
// kernels hold theirs, and frees them on both outcomes.
#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {
namespace {

__global__ void __launch_bounds__(32, 1) k_wait_check(uint32_t iters, int complete, int32_t *err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int lane = threadIdx.x;
  tc::tmem_alloc(&tmem_base, 32);
  tc::tmem_relinquish();
  if (lane == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  tc::tc_fence_before();
  __syncwarp();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (lane == 0 && complete) tc::mbar_arrive(&bar);
  int ok = 1;
  if (lane == 0) ok = tc::mbar_wait_bounded(&bar, 0, iters) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok && lane == 0) raise_err(err, CSA2_DEVERR_TIMEOUT);
  tc::tc_fence_before();
  __syncwarp();
  tc::tc_fence_after();
  tc::tmem_dealloc(tmem, 32);
}

}  // namespace
}  // namespace csa2

extern "C" csa2_status csa2_bounded_wait_check(int32_t iters, int32_t complete, int32_t *err_word,
                                               csa2_stream_t stream) {
  CSA2_REQUIRE(iters >= 1 && iters <= 64, CSA2_ERR_SHAPE, "iters %d outside 1..64", iters);
  CSA2_REQUIRE(complete == 0 || complete == 1, CSA2_ERR_RANGE, "complete %d is not 0 or 1", complete);
  CSA2_REQUIRE(err_word != nullptr, CSA2_ERR_NULL, "err_word is NULL");
  CSA2_REQUIRE((reinterpret_cast<uintptr_t>(err_word) & 3u) == 0, CSA2_ERR_ALIGN,
               "err_word is not 4-byte aligned");
  csa2::k_wait_check<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<uint32_t>(iters), complete,
                                                                            err_word);
  return csa2::cuda_status(cudaGetLastError(), "csa2_bounded_wait_check");
}
