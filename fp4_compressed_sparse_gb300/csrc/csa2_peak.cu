// csa2_peak.cu -- dense throughput of the block-scaled FP4 tensor-core MMA that
// the index score uses (tcgen05.mma kind::mxf4, E2M1 x E2M1 with UE8M0 scales,
// fp32 accumulate), measured with operands resident in shared memory.
//
// The indexer QK product runs in FP4 ([P5] "DeepSeek-V4: Towards Highly
// Efficient Million-Token Context Intelligence" §2.3.4); the prefill indexer is
// a dense contraction whose tensor-pipe utilisation is reported against this
// measured rate.  One CTA per SM; one thread issues back-to-back MMAs of shape
// M 128 x N 128 x K 64 (the score kernel's shape at 128 heads) into two TMEM
// accumulators, with no memory traffic, then waits (bounded) for the last one.
// The caller times the launch; each CTA does iters x 2 x 128 x 128 x 64 FLOP.
#include "csa2_internal.cuh"
#include "csa2_tc.cuh"

namespace csa2 {
namespace {

constexpr int kPeakN = 128;
constexpr uint32_t kPeakWaitIters = 2000;  // suspended polls of <= 1 ms each

__global__ void __launch_bounds__(128, 1) k_mxf4_peak(int iters, uint32_t *sink, int32_t *err) {
  __shared__ __align__(1024) uint8_t a_tile[kIdxTileCodeBytes];   // 128 rows x 128 E2M1 values
  __shared__ __align__(1024) uint8_t b_tile[kPeakN * 64];          // 128 rows x 128 E2M1 values
  __shared__ __align__(128) uint8_t sfa[512], sfb[512];            // one UE8M0 per 32 values (1.0)
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x;
  uint32_t x = 0x9E3779B9u * (tid + 1) + blockIdx.x;
  for (int i = tid; i < kIdxTileCodeBytes / 4; i += blockDim.x) {
    x = x * 1664525u + 1013904223u;
    reinterpret_cast<uint32_t *>(a_tile)[i] = x;
  }
  for (int i = tid; i < kPeakN * 64 / 4; i += blockDim.x) {
    x = x * 1664525u + 1013904223u;
    reinterpret_cast<uint32_t *>(b_tile)[i] = x;
  }
  for (int i = tid; i < 512; i += blockDim.x) sfa[i] = sfb[i] = 127;
  tc::fence_proxy_async_smem();  // generic writes, read by the tensor cores
  if (tid < 32) {
    tc::tmem_alloc(&tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&done, 1);
    tc::fence_mbar_init();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    const uint32_t col_sfa = 2 * kPeakN, col_sfb = 2 * kPeakN + 8;
    tc::tmem_cp_32x128b_x4(tmem + col_sfa, tc::smem_desc_noswizzle(tc::smem_addr(sfa), 128, 128));
    tc::tmem_cp_32x128b_x4(tmem + col_sfb, tc::smem_desc_noswizzle(tc::smem_addr(sfb), 128, 128));
    const uint32_t id0 = tc::idesc_mxf4(128, kPeakN, 0, 0), id1 = tc::idesc_mxf4(128, kPeakN, 2, 2);
    const uint32_t sa = tc::smem_addr(a_tile), sb = tc::smem_addr(b_tile);
    for (int i = 0; i < iters; ++i) {
      const int h = i & 1;  // K half: blocks 0-1 or 2-3 of the 128-value rows
      tc::mma_mxf4(tmem + ((i >> 1) & 1) * kPeakN, tc::smem_desc_noswizzle(sa + 4096 * h, 2048, 128),
                   tc::smem_desc_noswizzle(sb + 2 * kPeakN * 16 * h, kPeakN * 16, 128), h ? id1 : id0,
                   tmem + col_sfa, tmem + col_sfb, i >= 2 ? 1u : 0u);
    }
    tc::mma_commit(&done);
  }
  __syncwarp();
  int ok = 1;
  if ((tid & 31) == 0) ok = tc::mbar_wait_bounded(&done, 0, kPeakWaitIters) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok && tid == 0) raise_err(err, CSA2_DEVERR_TIMEOUT);
  tc::tc_fence_after();
  uint32_t v = 0;
  if (ok) {
    tc::tmem_ld_32x32b_x1(tmem + (static_cast<uint32_t>(32 * (tid >> 5)) << 16), v);
    tc::tmem_ld_wait();
    asm volatile("" : "+r"(v));
  }
  if (tid == 0 && sink) sink[blockIdx.x] = v;  // keeps the result observable
  tc::tc_fence_before();
  __syncthreads();
  if (tid < 32) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace
}  // namespace csa2

extern "C" csa2_status csa2_mxf4_peak_launch(int32_t n_ctas, int32_t iters, uint32_t *sink, int32_t *err_word,
                                             csa2_stream_t stream) {
  CSA2_REQUIRE(n_ctas >= 1 && n_ctas <= 4096, CSA2_ERR_SHAPE, "n_ctas %d outside 1..4096", n_ctas);
  CSA2_REQUIRE(iters >= 2 && iters <= (1 << 24), CSA2_ERR_SHAPE, "iters %d outside 2..2^24", iters);
  CSA2_REQUIRE_OPT_PTR(sink);
  csa2::k_mxf4_peak<<<n_ctas, 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(iters, sink, err_word);
  return csa2::cuda_status(cudaGetLastError(), "csa2_mxf4_peak_launch");
}
