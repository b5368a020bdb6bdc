// csa2_internal.cuh -- launchers shared between the libcsa2 translation units.
#pragma once

#include "csa2_device.cuh"

namespace csa2 {

// ------------------------------------------------------------------ host helpers (csa2_api.cu)
// thread-local text returned by csa2_last_error_detail()
void set_error_detail(const char *msg);
// records a printf-style detail for csa2_last_error_detail() and returns st
csa2_status fail(csa2_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
// CSA2_OK for cudaSuccess, else CSA2_ERR_CUDA with "what: <CUDA error text>" as the detail
csa2_status cuda_status(cudaError_t e, const char *what);
// SM count of the current device (queried once per device)
int device_sm_count();
// Raises fn's dynamic shared-memory limit to at least `bytes` on the current
// device (the attribute is per device: set once per (device, kernel)).
cudaError_t ensure_smem_limit(const void *fn, int bytes);

__host__ __forceinline__ bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define CSA2_REQUIRE(cond, status, ...)                  \
  do {                                                   \
    if (!(cond)) return ::csa2::fail(status, __VA_ARGS__); \
  } while (0)

#define CSA2_REQUIRE_PTR(p)                                                                 \
  do {                                                                                      \
    if ((p) == nullptr) return ::csa2::fail(CSA2_ERR_NULL, "%s is NULL", #p);               \
    if (!::csa2::aligned16(p)) return ::csa2::fail(CSA2_ERR_ALIGN, "%s is not 16-byte aligned", #p); \
  } while (0)

#define CSA2_REQUIRE_OPT_PTR(p)                                                             \
  do {                                                                                      \
    if ((p) != nullptr && !::csa2::aligned16(p))                                            \
      return ::csa2::fail(CSA2_ERR_ALIGN, "%s is not 16-byte aligned", #p);                 \
  } while (0)

cudaError_t launch_kv_append(const csa2_cache &c, const void *kv, const void *ik, int in_dtype,
                             const csa2_compress_in *cmp, const float *rope_cs, int64_t rope_len, int n_new,
                             float *cmp_dbg, int32_t *err, cudaStream_t s);

// ------------------------------------------------------------------ score sideband
// Per score row, the index-score kernel also leaves a 13-bit histogram of the
// order-preserving score keys and (FULL rows) the maxima of 8-position blocks
// with their histogram; the selector reads these instead of re-scanning.
// Row layout: hist[0][kSelBins] (scores) | hist[1][kSelBins] (block maxima) |
// bmax[ceil(stride/8)] floats, padded to 16 bytes.
constexpr int kSelBins = 8192;
constexpr int kSelBinShift = 19;  // key >> 19 = top 13 bits
constexpr int kSelCap = 4096;     // candidates kept per (row, problem)
__host__ __device__ __forceinline__ int64_t aux_row_bytes(int64_t stride) {
  return 2 * kSelBins * 4 + ((((stride + 7) / 8) * 4 + 15) / 16) * 16;
}

// ------------------------------------------------------------------ index score
struct ScoreArgs {
  const uint8_t *idx_codes;   // cache plane base
  const uint8_t *idx_scales;
  EntryMap map;               // where a sequence's entries live (dense or paged)
  int64_t cap;                // entries per sequence
  int ratio;
  int rows;                   // query rows
  int heads;                  // H_I
  const uint16_t *q_idx;      // [rows][H_I][128] bf16
  const float *w;             // [rows][H_I]
  const int64_t *q_pos;       // [rows]
  int cache_seq;              // -1: row r reads sequence r; else every row reads this sequence
  const int32_t *pool;        // POOL mode: [rows][pool_blocks]; nullptr = FULL
  int pool_blocks, pool_bs;
  float *scores;              // [rows][stride]
  int64_t stride;
  uint8_t *aux;               // [rows][aux_row_bytes(stride)] sideband (its histograms are cleared by the launch), or nullptr
  int32_t *err;
  int no_block_max;           // FULL with aux: 1 = the score histogram alone (no pool will be built from it)
};
cudaError_t launch_index_score(const ScoreArgs &a, cudaStream_t s);  // CUDA cores (dp4a), no sideband
// tensor cores (tcgen05 kind::mxf4); needs pool == nullptr or pool_bs == 8, heads <= 128; fills aux
size_t score_tc_workspace_bytes(int rows, int heads);
cudaError_t launch_index_score_tc(const ScoreArgs &a, void *ws, cudaStream_t s);

// ------------------------------------------------------------------ top-k
struct TopkArgs {
  int rows;
  const float *scores;        // [rows][stride]
  int64_t stride;
  const uint8_t *aux;         // sideband from the score kernel, or nullptr (built here)
  int ratio;
  const int64_t *q_pos;       // [rows]
  const int32_t *pool;        // POOL rows: [rows][pool_blocks] ascending block ids; nullptr = FULL
  int pool_blocks, bs;
  int k;
  int32_t *idx_out;           // [rows][k]
  int out_pool_blocks;        // FULL only: candidate-pool size (0 = no pool)
  int32_t *pool_out;          // [rows][out_pool_blocks]
  int32_t *pool_count;        // [rows]
  int32_t *err;
};
size_t topk_workspace_bytes(int rows, int64_t stride, bool have_aux);
// fills the sideband of `rows` score rows from the scores themselves
cudaError_t launch_fill_aux(const TopkArgs &a, uint8_t *aux, cudaStream_t s);
cudaError_t launch_topk(const TopkArgs &a, void *ws, cudaStream_t s);

// ------------------------------------------------------------------ attention
struct AttnArgs {
  int rows, heads, k;
  const uint16_t *q;          // [rows][H][576]
  const int32_t *idx;         // [rows][k]
  const int64_t *q_pos;       // [rows]
  int cache_seq;              // -1: row = sequence
  const uint8_t *lat_codes, *lat_scales, *rope_codes, *rope_scales;
  EntryMap map;               // where a sequence's entries live (dense or paged)
  int entry_format;           // CSA2_ENTRY_FP4 or CSA2_ENTRY_FP8
  int64_t cap;
  int ratio;
  const int64_t *n_tokens;    // [batch]
  const uint8_t *ring_codes, *ring_scales;  // window ring [seq][128][...]
  int ring_single;            // 1: the ring holds only cache_seq's 128 slots
  int swa_dtype;
  const uint8_t *lin_codes, *lin_scales;    // window tokens >= *lin_base: [t - *lin_base][...]
  const int64_t *lin_base;    // device scalar or nullptr
  const float *sink;          // [H] or nullptr
  float sm_scale;
  float *out, *lse;
  int32_t *err;
};
// Segments of a decode row (a function of k alone: the batch-invariant
// accumulation order); a row's output is the ordered merge of its segments.
int attn_segments(int k);
size_t attn_workspace_bytes(int rows, int heads, int n_seg);
cudaError_t launch_attn(const AttnArgs &a, int n_seg, void *ws, size_t ws_bytes, cudaStream_t s);

}  // namespace csa2
