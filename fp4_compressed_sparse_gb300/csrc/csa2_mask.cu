// csa2_mask.cu -- the Reindex selection in the form of the public reference
// code: every visible position scored (FULL), then every position outside the
// candidate pool masked to -inf, then the top-k of the whole row.
//
// [P1] "DeepSeek V4.1 Flash 아키텍처 분석", §"공개 코드를 읽어 보니 남는 차이":
// the published Indexer.forward computes the scores of all keys and masks the
// ones outside the candidates; the Hierarchical Sparse Indexer's saving
// (§"512개를 고르기 위해 ...": a Reindex layer scores only its 2,048 x 8 pool
// positions) is that this full scan is not needed.  This file exists for the
// comparison of the two forms; the selected positions agree whenever the pool
// holds at least k visible positions.
//
// One thread per pool-block-sized group of positions: a binary search for the
// group's block id in the row's ascending pool, and -inf over the group when it
// is absent.
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

__global__ void __launch_bounds__(256) k_mask_to_pool(float *scores, int64_t stride, int ratio, const int64_t *q_pos,
                                                      const int32_t *pool, int pool_blocks, int bs) {
  const int row = blockIdx.y;
  int64_t T = q_pos[row] / ratio;
  if (T < 0) T = 0;
  if (T > stride) T = stride;
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (blk * bs >= T) return;
  const int32_t *p = pool + static_cast<size_t>(row) * pool_blocks;
  // ascending ids, -1 padding at the end: the valid prefix ends at the first -1
  int lo = 0, hi = pool_blocks;  // search [lo, hi) for blk
  bool found = false;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int32_t v = __ldg(p + mid);
    if (v == blk) {
      found = true;
      break;
    }
    if (v < 0 || v > blk) hi = mid;
    else lo = mid + 1;
  }
  if (found) return;
  float *s = scores + static_cast<size_t>(row) * stride;
  const int64_t e = min(T, (blk + 1) * bs);
  for (int64_t i = blk * bs; i < e; ++i) s[i] = -INFINITY;
}

}  // namespace
}  // namespace csa2

extern "C" csa2_status csa2_mask_to_pool(float *scores, int64_t score_stride, int32_t batch, int32_t ratio,
                                         const int64_t *q_pos, const int32_t *pool, int32_t pool_blocks,
                                         int32_t pool_block_size, csa2_stream_t stream) {
  CSA2_REQUIRE_PTR(scores);
  CSA2_REQUIRE_PTR(q_pos);
  CSA2_REQUIRE_PTR(pool);
  CSA2_REQUIRE(batch >= 1 && batch <= 65535, CSA2_ERR_SHAPE, "batch %d outside 1..65535", batch);
  CSA2_REQUIRE(ratio == 1 || ratio == 2, CSA2_ERR_RANGE, "ratio %d (must be 1 or 2)", ratio);
  CSA2_REQUIRE(score_stride >= 1, CSA2_ERR_SHAPE, "score_stride %lld < 1", static_cast<long long>(score_stride));
  CSA2_REQUIRE(pool_blocks >= 1 && pool_blocks <= (1 << 24), CSA2_ERR_SHAPE, "pool_blocks %d", pool_blocks);
  CSA2_REQUIRE(pool_block_size >= 1 && pool_block_size <= 64, CSA2_ERR_SHAPE, "pool_block_size %d outside 1..64",
               pool_block_size);
  const int64_t groups = (score_stride + pool_block_size - 1) / pool_block_size;
  const dim3 grid(static_cast<unsigned>((groups + 255) / 256), static_cast<unsigned>(batch));
  csa2::k_mask_to_pool<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      scores, score_stride, ratio, q_pos, pool, pool_blocks, pool_block_size);
  return csa2::cuda_status(cudaGetLastError(), "csa2_mask_to_pool launch");
}
