// csa2_internal.cuh -- launchers shared between the libcsa2 translation units.
#pragma once

#include "csa2_device.cuh"

namespace csa2 {

// thread-local text returned by csa2_last_error_detail()
void set_error_detail(const char *msg);

cudaError_t launch_kv_append(const csa2_cache &c, const void *kv, const void *ik, int in_dtype,
                             const csa2_compress_in *cmp, const float *rope_cs, int64_t rope_len, int n_new,
                             float *cmp_dbg, int32_t *err, cudaStream_t s);

// ------------------------------------------------------------------ index score
struct ScoreArgs {
  const uint8_t *idx_codes;   // cache plane base
  const uint8_t *idx_scales;
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
  int32_t *err;
};
cudaError_t launch_index_score(const ScoreArgs &a, cudaStream_t s);  // CUDA cores (dp4a)
// tensor cores (tcgen05 kind::mxf4); needs pool == nullptr or pool_bs == 8, heads <= 128
size_t score_tc_workspace_bytes(int rows, int heads);
cudaError_t launch_index_score_tc(const ScoreArgs &a, void *ws, cudaStream_t s);

// ------------------------------------------------------------------ top-k
enum SelMode { kSelFull = 0, kSelPool = 1, kSelBlockMax = 2 };
struct SelArgs {
  int rows;
  const float *scores;
  int64_t stride;
  int ratio;
  const int64_t *q_pos;
  const int32_t *pool;  // kSelPool
  int pool_blocks, bs;
  int mode;
  int k;
  int32_t *out;         // [rows][out_stride]
  int out_stride;
  int32_t *count_out;   // [rows] or nullptr
  int32_t *err;
};
size_t select_workspace_bytes(int rows, int64_t max_slots);
cudaError_t launch_select(const SelArgs &a, int64_t max_slots, void *ws, cudaStream_t s);

// ------------------------------------------------------------------ attention
struct AttnArgs {
  int rows, heads, k;
  const uint16_t *q;          // [rows][H][576]
  const int32_t *idx;         // [rows][k]
  const int64_t *q_pos;       // [rows]
  int cache_seq;              // -1: row = sequence
  const uint8_t *lat_codes, *lat_scales, *rope_codes, *rope_scales;
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
  float *part;                // split partials
  int32_t *err;
};
size_t attn_workspace_bytes(int rows, int heads, int k);
cudaError_t launch_attn(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t s);

}  // namespace csa2
