// csa2_api.cu -- the libcsa2 C ABI: host-side validation, workspace sizing and
// launches.  See include/csa2.h for the contract of every entry point.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "csa2_encode.cuh"
#include "csa2_internal.cuh"

namespace {

thread_local std::string g_detail;

// Optional phase markers of this thread's next csa2_prefill_chunk calls
// (csa2_set_phase_events): events recorded on the call's stream in order.
thread_local cudaEvent_t *g_phase_ev = nullptr;
thread_local int g_phase_cap = 0, g_phase_used = 0;

void mark_phase(cudaStream_t s) {
  if (g_phase_ev != nullptr && g_phase_used < g_phase_cap) cudaEventRecord(g_phase_ev[g_phase_used++], s);
}

}  // namespace

namespace csa2 {

void set_error_detail(const char *msg) { g_detail = msg ? msg : ""; }

csa2_status fail(csa2_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_detail = buf;
  return st;
}

csa2_status cuda_status(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return CSA2_OK;
  return fail(CSA2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int g_sm_count[kMaxDevices] = {};
std::map<std::pair<int, const void *>, int> g_smem_limit;  // (device, kernel) -> bytes set
}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  if (dev >= 0 && dev < kMaxDevices) {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (g_sm_count[dev] > 0) return g_sm_count[dev];
  }
  int n = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // a failed query is not sticky: clear it so the next launch reports its own status
    return 1;
  }
  if (dev < kMaxDevices) {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    g_sm_count[dev] = n;
  }
  return n;
}

cudaError_t ensure_smem_limit(const void *fn, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_pair(dev, fn);
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    auto it = g_smem_limit.find(key);
    if (it != g_smem_limit.end() && it->second >= bytes) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  int &have = g_smem_limit[key];
  if (bytes > have) have = bytes;
  return cudaSuccess;
}

}  // namespace csa2

namespace {

using csa2::aligned16;
using csa2::cuda_status;
using csa2::fail;

#define REQUIRE CSA2_REQUIRE
#define REQUIRE_PTR CSA2_REQUIRE_PTR
#define REQUIRE_OPT_PTR CSA2_REQUIRE_OPT_PTR

csa2_status check_cache(const csa2_cache *c) {
  REQUIRE(c != nullptr, CSA2_ERR_NULL, "cache is NULL");
  REQUIRE(c->batch >= 1 && c->batch <= 65535, CSA2_ERR_SHAPE, "cache batch %d outside 1..65535", c->batch);
  REQUIRE(c->capacity >= 1 && c->capacity <= (1 << 30), CSA2_ERR_SHAPE, "cache capacity %d outside 1..2^30",
          c->capacity);
  REQUIRE(c->ratio == 1 || c->ratio == 2, CSA2_ERR_RANGE, "cache ratio %d (must be 1 or 2)", c->ratio);
  REQUIRE(c->swa_dtype == CSA2_SWA_BF16 || c->swa_dtype == CSA2_SWA_MXFP8, CSA2_ERR_RANGE, "swa_dtype %d",
          c->swa_dtype);
  REQUIRE(c->entry_format == CSA2_ENTRY_FP4 || c->entry_format == CSA2_ENTRY_FP8, CSA2_ERR_RANGE,
          "entry_format %d", c->entry_format);
  REQUIRE_PTR(c->lat_codes);
  REQUIRE_PTR(c->lat_scales);
  REQUIRE_PTR(c->rope_codes);
  if (c->entry_format == CSA2_ENTRY_FP4) REQUIRE_PTR(c->rope_scales);
  REQUIRE_PTR(c->idx_codes);
  REQUIRE_PTR(c->idx_scales);
  REQUIRE_PTR(c->swa_codes);
  if (c->swa_dtype == CSA2_SWA_MXFP8) REQUIRE_PTR(c->swa_scales);
  REQUIRE_PTR(c->n_tokens);
  if (c->ratio == 2) REQUIRE_PTR(c->cmp_buf);
  if (c->block_table != nullptr) {
    REQUIRE_PTR(c->block_table);
    REQUIRE(c->page_entries >= 128 && c->page_entries % 128 == 0, CSA2_ERR_SHAPE,
            "page_entries %d must be a positive multiple of 128", c->page_entries);
    REQUIRE(c->max_pages >= 1 && c->n_pages >= 1, CSA2_ERR_SHAPE, "max_pages %d / n_pages %d", c->max_pages,
            c->n_pages);
    REQUIRE(static_cast<int64_t>(c->max_pages) * c->page_entries == c->capacity, CSA2_ERR_SHAPE,
            "capacity %d != max_pages %d x page_entries %d", c->capacity, c->max_pages, c->page_entries);
  }
  return CSA2_OK;
}

// A view of one sequence of a cache (batch 1).
csa2_cache seq_view(const csa2_cache &c, int seq) {
  csa2_cache v = c;
  v.batch = 1;
  if (c.block_table != nullptr) {
    v.block_table += static_cast<size_t>(seq) * c.max_pages;  // the entry planes are the shared page pool
  } else {
    const size_t e = static_cast<size_t>(seq) * c.capacity;
    v.lat_codes += e * csa2_entry_plane_bytes(c.entry_format, 0);
    v.lat_scales += e * csa2_entry_plane_bytes(c.entry_format, 1);
    v.rope_codes += e * csa2_entry_plane_bytes(c.entry_format, 2);
    if (v.rope_scales) v.rope_scales += e * csa2_entry_plane_bytes(c.entry_format, 3);
    v.idx_codes += static_cast<size_t>(seq) * csa2::idx_tiles(c.capacity) * csa2::kIdxTileCodeBytes;
    v.idx_scales += static_cast<size_t>(seq) * csa2::idx_tiles(c.capacity) * csa2::kIdxTileScaleBytes;
  }
  v.swa_codes += static_cast<size_t>(seq) * csa2::kWin * (c.swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152);
  if (v.swa_scales) v.swa_scales += static_cast<size_t>(seq) * csa2::kWin * csa2::kSwaScaleStride;
  if (v.cmp_buf) v.cmp_buf += static_cast<size_t>(seq) * 4 * 4 * csa2::kDcmp;
  v.n_tokens += seq;
  return v;
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

// ===================================================================== prefill kernels
namespace csa2 {
namespace {

// P = n_tokens (before the append), q_pos[i] = P + i, and a copy of the window ring.
__global__ void k_prefill_snapshot(csa2_cache v, int Q, int64_t *P, int64_t *q_pos, uint8_t *ring_codes,
                                   uint8_t *ring_scales) {
  const int64_t p0 = v.n_tokens[0];
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  if (tid == 0) *P = p0;
  for (int i = tid; i < Q; i += gridDim.x * blockDim.x) q_pos[i] = p0 + i;
  const int cb = v.swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152;
  const int n16 = kWin * cb / 16;
  for (int i = tid; i < n16; i += gridDim.x * blockDim.x)
    reinterpret_cast<uint4 *>(ring_codes)[i] = reinterpret_cast<const uint4 *>(v.swa_codes)[i];
  if (v.swa_scales)
    for (int i = tid; i < kWin * kSwaScaleStride / 16; i += gridDim.x * blockDim.x)
      reinterpret_cast<uint4 *>(ring_scales)[i] = reinterpret_cast<const uint4 *>(v.swa_scales)[i];
}

// Window rows of every chunk token: its own C^a[0:576], rotated at P+i.
__global__ void __launch_bounds__(256) k_prefill_window(const float *ca, int Q, const int64_t *P, const float *rope_cs,
                                                        int64_t rope_len, int swa_dtype, uint8_t *lin_codes,
                                                        uint8_t *lin_scales) {
  __shared__ float srow[8][kDqk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + warp;
  if (i >= Q) return;
  const int64_t t = *P + i;
  if (t >= rope_len) return;  // the append reports the ROPE error
  for (int d = lane; d < kDqk; d += 32) srow[warp][d] = ca[static_cast<size_t>(i) * kDcmp + d];
  __syncwarp();
  const int cb = swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152;
  warp_encode_swa(lin_codes + static_cast<size_t>(i) * cb,
                  lin_scales ? lin_scales + static_cast<size_t>(i) * kSwaScaleStride : nullptr, swa_dtype,
                  srow[warp], rope_cs + t * 64, lane);
}

}  // namespace
}  // namespace csa2

// ===================================================================== C ABI
extern "C" {

int32_t csa2_version(void) { return 200; }

const char *csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_NULL: return "a required pointer is NULL";
    case CSA2_ERR_SHAPE: return "a size is outside its documented range";
    case CSA2_ERR_ALIGN: return "a device pointer is not 16-byte aligned";
    case CSA2_ERR_RANGE: return "an argument is out of range";
    case CSA2_ERR_UNSUPPORTED: return "not supported";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

const char *csa2_last_error_detail(void) { return g_detail.c_str(); }

csa2_status csa2_set_phase_events(void *const *events, int32_t n_events) {
  REQUIRE(n_events >= 0, CSA2_ERR_SHAPE, "n_events %d < 0", n_events);
  REQUIRE(n_events == 0 || events != nullptr, CSA2_ERR_NULL, "events is NULL");
  g_phase_ev = n_events ? reinterpret_cast<cudaEvent_t *>(const_cast<void **>(events)) : nullptr;
  g_phase_cap = n_events;
  g_phase_used = 0;
  return CSA2_OK;
}

int32_t csa2_phase_events_recorded(void) { return g_phase_used; }

size_t csa2_cache_plane_bytes(int32_t batch, int32_t capacity, int32_t plane, int32_t swa_dtype) {
  const size_t e = static_cast<size_t>(batch) * capacity;
  switch (plane) {
    case 0: return e * 256;
    case 1: return e * 32;
    case 2: return e * 32;
    case 3: return e * 4;
    case 4: return static_cast<size_t>(batch) * csa2::idx_tiles(capacity) * csa2::kIdxTileCodeBytes;
    case 5: return static_cast<size_t>(batch) * csa2::idx_tiles(capacity) * csa2::kIdxTileScaleBytes;
    case 6: return static_cast<size_t>(batch) * csa2::kWin * (swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152);
    case 7: return static_cast<size_t>(batch) * csa2::kWin * csa2::kSwaScaleStride;
    case 8: return static_cast<size_t>(batch) * 4 * 4 * csa2::kDcmp * sizeof(float);
    case 9: return static_cast<size_t>(batch) * sizeof(int64_t);
  }
  return 0;
}

size_t csa2_entry_plane_bytes(int32_t entry_format, int32_t plane) {
  static const size_t fp4[6] = {256, 32, 32, 4, 64, 4}, fp8[6] = {512, 16, 128, 0, 64, 4};
  if (plane < 0 || plane > 5) return 0;
  if (entry_format == CSA2_ENTRY_FP4) return fp4[plane];
  if (entry_format == CSA2_ENTRY_FP8) return fp8[plane];
  return 0;
}

size_t csa2_paged_plane_bytes(int32_t n_pages, int32_t page_entries, int32_t plane) {
  if (n_pages <= 0 || page_entries <= 0 || page_entries % 128 != 0) return 0;
  const size_t e = static_cast<size_t>(n_pages) * page_entries;
  switch (plane) {
    case 0: return e * 256;
    case 1: return e * 32;
    case 2: return e * 32;
    case 3: return e * 4;
    case 4: return e / csa2::kIdxTile * csa2::kIdxTileCodeBytes;
    case 5: return e / csa2::kIdxTile * csa2::kIdxTileScaleBytes;
  }
  return 0;
}

csa2_status csa2_rope_table(double theta, int64_t n_pos, float *out_host) {
  REQUIRE(out_host != nullptr, CSA2_ERR_NULL, "out_host is NULL");
  REQUIRE(n_pos >= 0, CSA2_ERR_SHAPE, "n_pos %lld < 0", static_cast<long long>(n_pos));
  REQUIRE(theta > 0.0, CSA2_ERR_RANGE, "theta must be > 0");
  double inv_freq[csa2::kRope / 2];
  for (int i = 0; i < csa2::kRope / 2; ++i) inv_freq[i] = std::pow(theta, -static_cast<double>(2 * i) / csa2::kRope);
  for (int64_t p = 0; p < n_pos; ++p)
    for (int i = 0; i < csa2::kRope / 2; ++i) {
      const double ang = static_cast<double>(p) * inv_freq[i];
      out_host[p * 64 + 2 * i] = static_cast<float>(std::cos(ang));
      out_host[p * 64 + 2 * i + 1] = static_cast<float>(std::sin(ang));
    }
  return CSA2_OK;
}

csa2_status csa2_kv_append(const csa2_cache *cache, const void *kv, const void *idx_key, int32_t in_dtype,
                           const csa2_compress_in *cmp, const float *rope_cs, int64_t rope_len, int32_t n_new,
                           float *cmp_dbg, int32_t *err_word, csa2_stream_t stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  REQUIRE(n_new >= 0, CSA2_ERR_SHAPE, "n_new %d < 0", n_new);
  REQUIRE_PTR(rope_cs);
  REQUIRE(rope_len >= 1, CSA2_ERR_SHAPE, "rope_len %lld < 1", static_cast<long long>(rope_len));
  REQUIRE_OPT_PTR(cmp_dbg);
  if (cache->ratio == 1) {
    REQUIRE(cmp == nullptr, CSA2_ERR_RANGE, "cmp must be NULL for a ratio-1 cache");
    REQUIRE(in_dtype == CSA2_IN_F32 || in_dtype == CSA2_IN_BF16, CSA2_ERR_RANGE, "in_dtype %d", in_dtype);
    REQUIRE_PTR(kv);
    REQUIRE_PTR(idx_key);
  } else {
    REQUIRE(cmp != nullptr, CSA2_ERR_NULL, "cmp is NULL for a ratio-2 cache");
    REQUIRE_PTR(cmp->ca);
    REQUIRE_PTR(cmp->cb);
    REQUIRE_PTR(cmp->za);
    REQUIRE_PTR(cmp->zb);
    REQUIRE_PTR(cmp->ba);
    REQUIRE_PTR(cmp->bb);
  }
  if (n_new == 0) return CSA2_OK;
  return cuda_status(csa2::launch_kv_append(*cache, kv, idx_key, in_dtype, cmp, rope_cs, rope_len, n_new, cmp_dbg,
                                            err_word, reinterpret_cast<cudaStream_t>(stream)),
                     "csa2_kv_append launch");
}

size_t csa2_index_score_workspace_size(int32_t batch, int32_t n_heads_idx) {
  if (batch <= 0 || n_heads_idx <= 0) return 256;
  return csa2::score_tc_workspace_bytes(batch, n_heads_idx);
}

size_t csa2_score_aux_size(int32_t batch, int64_t score_stride) {
  if (batch <= 0 || score_stride <= 0) return 256;
  return static_cast<size_t>(batch) * csa2::aux_row_bytes(score_stride);
}

csa2_status csa2_index_score(const csa2_cache *cache, const uint16_t *q_idx, const float *w, int32_t n_heads_idx,
                             const int64_t *q_pos, const int32_t *pool, int32_t pool_blocks,
                             int32_t pool_block_size, float *scores, int64_t score_stride, void *score_aux, void *ws,
                             size_t ws_bytes, int32_t *err_word, csa2_stream_t stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  REQUIRE_PTR(q_idx);
  REQUIRE_PTR(w);
  REQUIRE_PTR(q_pos);
  REQUIRE_PTR(scores);
  REQUIRE_OPT_PTR(score_aux);
  REQUIRE(n_heads_idx >= 1 && n_heads_idx <= CSA2_MAX_HEADS, CSA2_ERR_SHAPE, "n_heads_idx %d outside 1..128",
          n_heads_idx);
  if (pool) {
    REQUIRE_PTR(pool);
    REQUIRE(pool_blocks >= 1 && pool_block_size >= 1 && pool_block_size <= 64, CSA2_ERR_SHAPE,
            "pool_blocks %d / pool_block_size %d", pool_blocks, pool_block_size);
    REQUIRE(score_stride >= static_cast<int64_t>(pool_blocks) * pool_block_size, CSA2_ERR_SHAPE,
            "score_stride %lld < pool_blocks*pool_block_size", static_cast<long long>(score_stride));
  } else {
    REQUIRE(score_stride >= cache->capacity, CSA2_ERR_SHAPE, "score_stride %lld < capacity %d",
            static_cast<long long>(score_stride), cache->capacity);
  }
  csa2::ScoreArgs a{};
  a.idx_codes = cache->idx_codes;
  a.idx_scales = cache->idx_scales;
  a.map = csa2::entry_map(*cache);
  a.cap = cache->capacity;
  a.ratio = cache->ratio;
  a.rows = cache->batch;
  a.heads = n_heads_idx;
  a.q_idx = q_idx;
  a.w = w;
  a.q_pos = q_pos;
  a.cache_seq = -1;
  a.pool = pool;
  a.pool_blocks = pool_blocks;
  a.pool_bs = pool_block_size;
  a.scores = scores;
  a.stride = score_stride;  // row stride of scores in both modes
  a.aux = static_cast<uint8_t *>(score_aux);
  a.err = err_word;
  const size_t need = csa2_index_score_workspace_size(cache->batch, n_heads_idx);
  REQUIRE(ws != nullptr && ws_bytes >= need, CSA2_ERR_WORKSPACE, "index-score workspace %zu < %zu bytes", ws_bytes,
          need);
  REQUIRE(aligned16(ws), CSA2_ERR_ALIGN, "ws is not 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (pool && pool_block_size != 8) {
    // CUDA-core path; the sideband is then built from the scores
    a.aux = nullptr;
    cudaError_t e = csa2::launch_index_score(a, s);
    if (e != cudaSuccess || !score_aux) return cuda_status(e, "csa2_index_score launch");
    csa2::TopkArgs t{};
    t.rows = cache->batch;
    t.scores = scores;
    t.stride = score_stride;
    t.ratio = cache->ratio;
    t.q_pos = q_pos;
    t.pool = pool;
    t.pool_blocks = pool_blocks;
    t.bs = pool_block_size;
    t.err = err_word;
    return cuda_status(csa2::launch_fill_aux(t, static_cast<uint8_t *>(score_aux), s), "csa2_index_score sideband");
  }
  return cuda_status(csa2::launch_index_score_tc(a, ws, s), "csa2_index_score launch");
}

size_t csa2_topk_workspace_size(int32_t batch, int64_t score_stride, int32_t k, int32_t out_pool_blocks) {
  (void)k;
  (void)out_pool_blocks;
  if (batch <= 0 || score_stride <= 0) return 256;
  return csa2::topk_workspace_bytes(batch, score_stride, false);
}

csa2_status csa2_topk(const float *scores, int64_t score_stride, const void *score_aux, int32_t batch, int32_t ratio,
                      const int64_t *q_pos, const int32_t *pool, int32_t pool_blocks, int32_t pool_block_size,
                      int32_t k, int32_t *idx_out, int32_t out_pool_blocks, int32_t *pool_out, int32_t *pool_count,
                      void *ws, size_t ws_bytes, int32_t *err_word, csa2_stream_t stream) {
  REQUIRE_PTR(scores);
  REQUIRE_OPT_PTR(score_aux);
  REQUIRE_PTR(q_pos);
  REQUIRE_PTR(idx_out);
  REQUIRE(batch >= 1 && batch <= 65535, CSA2_ERR_SHAPE, "batch %d", batch);
  REQUIRE(ratio == 1 || ratio == 2, CSA2_ERR_RANGE, "ratio %d", ratio);
  REQUIRE(k >= 1 && k <= CSA2_MAX_TOPK, CSA2_ERR_RANGE, "k %d outside 1..2048", k);
  REQUIRE(score_stride >= 1, CSA2_ERR_SHAPE, "score_stride %lld", static_cast<long long>(score_stride));
  REQUIRE(pool_block_size >= 1 && pool_block_size <= 64, CSA2_ERR_SHAPE, "pool_block_size %d", pool_block_size);
  if (pool) {
    REQUIRE_PTR(pool);
    REQUIRE(pool_blocks >= 1, CSA2_ERR_SHAPE, "pool_blocks %d", pool_blocks);
    REQUIRE(pool_out == nullptr, CSA2_ERR_RANGE, "a pool can only be built in FULL mode");
    REQUIRE(score_stride >= static_cast<int64_t>(pool_blocks) * pool_block_size, CSA2_ERR_SHAPE,
            "score_stride too small for the pool");
  }
  if (pool_out) {
    REQUIRE_PTR(pool_out);
    REQUIRE_PTR(pool_count);
    REQUIRE(out_pool_blocks >= 1 && out_pool_blocks <= CSA2_MAX_TOPK, CSA2_ERR_RANGE,
            "out_pool_blocks %d outside 1..2048", out_pool_blocks);
    REQUIRE(pool_block_size == 8, CSA2_ERR_UNSUPPORTED, "the candidate pool is built from 8-position blocks");
  }
  const size_t need = csa2::topk_workspace_bytes(batch, score_stride, score_aux != nullptr);
  REQUIRE(ws != nullptr && ws_bytes >= need, CSA2_ERR_WORKSPACE, "topk workspace %zu < %zu bytes", ws_bytes, need);
  REQUIRE(aligned16(ws), CSA2_ERR_ALIGN, "ws is not 16-byte aligned");
  csa2::TopkArgs a{};
  a.rows = batch;
  a.scores = scores;
  a.stride = score_stride;
  a.aux = static_cast<const uint8_t *>(score_aux);
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
  return cuda_status(csa2::launch_topk(a, ws, reinterpret_cast<cudaStream_t>(stream)), "csa2_topk launch");
}

size_t csa2_attn_workspace_size(int32_t batch, int32_t n_heads, int32_t k) {
  if (batch <= 0 || n_heads <= 0 || k <= 0) return 256;
  return csa2::attn_workspace_bytes(batch, n_heads, csa2::attn_segments(k));
}

csa2_status csa2_sparse_attn_decode(const csa2_cache *cache, const uint16_t *q, int32_t n_heads, const int64_t *q_pos,
                                    const int32_t *idx, int32_t k, const float *sink, float sm_scale, float *out,
                                    float *lse, void *ws, size_t ws_bytes, int32_t *err_word, csa2_stream_t stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  REQUIRE_PTR(q);
  REQUIRE_PTR(q_pos);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(out);
  REQUIRE_PTR(lse);
  REQUIRE_OPT_PTR(sink);
  REQUIRE(n_heads >= 16 && n_heads <= CSA2_MAX_HEADS && n_heads % 16 == 0, CSA2_ERR_SHAPE,
          "n_heads %d must be a multiple of 16 in 16..128", n_heads);
  REQUIRE(k >= 1 && k <= CSA2_MAX_TOPK, CSA2_ERR_RANGE, "k %d outside 1..2048", k);
  REQUIRE(std::isfinite(sm_scale), CSA2_ERR_RANGE, "sm_scale is not finite");
  const size_t need = csa2_attn_workspace_size(cache->batch, n_heads, k);
  REQUIRE(ws != nullptr && ws_bytes >= need, CSA2_ERR_WORKSPACE, "attention workspace %zu < %zu bytes", ws_bytes,
          need);
  REQUIRE(aligned16(ws), CSA2_ERR_ALIGN, "ws is not 16-byte aligned");
  csa2::AttnArgs a{};
  a.rows = cache->batch;
  a.heads = n_heads;
  a.k = k;
  a.q = q;
  a.idx = idx;
  a.q_pos = q_pos;
  a.cache_seq = -1;
  a.lat_codes = cache->lat_codes;
  a.lat_scales = cache->lat_scales;
  a.rope_codes = cache->rope_codes;
  a.rope_scales = cache->rope_scales;
  a.map = csa2::entry_map(*cache);
  a.entry_format = cache->entry_format;
  a.cap = cache->capacity;
  a.ratio = cache->ratio;
  a.n_tokens = cache->n_tokens;
  a.ring_codes = cache->swa_codes;
  a.ring_scales = cache->swa_scales;
  a.ring_single = 0;
  a.swa_dtype = cache->swa_dtype;
  a.lin_codes = nullptr;
  a.lin_scales = nullptr;
  a.lin_base = nullptr;
  a.sink = sink;
  a.sm_scale = sm_scale;
  a.out = out;
  a.lse = lse;
  a.err = err_word;
  return cuda_status(csa2::launch_attn(a, csa2::attn_segments(k), ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream)),
                     "csa2_sparse_attn_decode launch");
}

// -------------------------------------------------------------------- prefill
namespace {
struct PrefillLayout {
  int qb;  // queries per block
  size_t off_P, off_qpos, off_ring_c, off_ring_s, off_lin_c, off_lin_s, off_scores, off_aux, off_qrec, off_sel,
      off_attn, total;
};

PrefillLayout prefill_layout(int Q, int capacity, int n_heads, int k, int swa_dtype) {
  PrefillLayout L{};
  const int cb = swa_dtype == CSA2_SWA_MXFP8 ? 576 : 1152;
  // bound the score block to ~256 MB
  int qb = static_cast<int>((size_t(256) << 20) / (static_cast<size_t>(capacity) * 4));
  // whole waves: the attention runs one CTA per query and SM, the selection two
  // per SM, so a block of a multiple of 2 x SMs queries leaves no partial wave
  const int wave = 2 * csa2::device_sm_count();
  if (qb > wave) qb = qb / wave * wave;
  if (qb < 1) qb = 1;
  if (qb > Q) qb = Q;
  if (qb > 4096) qb = 4096;
  L.qb = qb;
  size_t o = 0;
  L.off_P = o;
  o = align256(o + 16);
  L.off_qpos = o;
  o = align256(o + static_cast<size_t>(Q) * 8);
  L.off_ring_c = o;
  o = align256(o + static_cast<size_t>(csa2::kWin) * cb);
  L.off_ring_s = o;
  o = align256(o + static_cast<size_t>(csa2::kWin) * csa2::kSwaScaleStride);
  L.off_lin_c = o;
  o = align256(o + static_cast<size_t>(Q) * cb);
  L.off_lin_s = o;
  o = align256(o + static_cast<size_t>(Q) * csa2::kSwaScaleStride);
  L.off_scores = o;
  o = align256(o + static_cast<size_t>(qb) * capacity * 4);
  L.off_aux = o;
  o = align256(o + static_cast<size_t>(qb) * csa2::aux_row_bytes(capacity));
  L.off_qrec = o;
  o = align256(o + csa2::score_tc_workspace_bytes(qb, 128));
  L.off_sel = o;
  o = align256(o + csa2::topk_workspace_bytes(qb, capacity, true));
  L.off_attn = o;
  o = align256(o + csa2::attn_workspace_bytes(qb, n_heads, 1));
  L.total = o;
  return L;
}
}  // namespace

size_t csa2_prefill_workspace_size(int32_t Q, int32_t capacity, int32_t n_heads_idx, int32_t n_heads, int32_t k) {
  (void)n_heads_idx;
  if (Q <= 0 || capacity <= 0 || n_heads <= 0 || k <= 0) return 256;
  // the window layout is sized for bf16 (the larger format)
  return prefill_layout(Q, capacity, n_heads, k, CSA2_SWA_BF16).total;
}

csa2_status csa2_prefill_chunk(const csa2_cache *cache, int32_t seq, const csa2_compress_in *cmp, const float *rope_cs,
                               int64_t rope_len, int32_t Q, const uint16_t *q_idx, const float *w,
                               int32_t n_heads_idx, const uint16_t *q, int32_t n_heads, int32_t k, const float *sink,
                               float sm_scale, int32_t *idx_out, float *out, float *lse, void *ws, size_t ws_bytes,
                               int32_t *err_word, csa2_stream_t stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  REQUIRE(cache->ratio == 2, CSA2_ERR_UNSUPPORTED, "csa2_prefill_chunk needs a ratio-2 cache");
  REQUIRE(seq >= 0 && seq < cache->batch, CSA2_ERR_RANGE, "seq %d outside the cache batch", seq);
  REQUIRE(cmp != nullptr, CSA2_ERR_NULL, "cmp is NULL");
  REQUIRE_PTR(cmp->ca);
  REQUIRE_PTR(cmp->cb);
  REQUIRE_PTR(cmp->za);
  REQUIRE_PTR(cmp->zb);
  REQUIRE_PTR(cmp->ba);
  REQUIRE_PTR(cmp->bb);
  REQUIRE_PTR(rope_cs);
  REQUIRE(Q >= 1 && Q <= (1 << 20), CSA2_ERR_SHAPE, "Q %d outside 1..2^20", Q);
  REQUIRE_PTR(q_idx);
  REQUIRE_PTR(w);
  REQUIRE_PTR(q);
  REQUIRE_PTR(idx_out);
  REQUIRE_PTR(out);
  REQUIRE_PTR(lse);
  REQUIRE_OPT_PTR(sink);
  REQUIRE(n_heads_idx >= 1 && n_heads_idx <= CSA2_MAX_HEADS, CSA2_ERR_SHAPE, "n_heads_idx %d", n_heads_idx);
  REQUIRE(n_heads >= 16 && n_heads <= CSA2_MAX_HEADS && n_heads % 16 == 0, CSA2_ERR_SHAPE, "n_heads %d", n_heads);
  REQUIRE(k >= 1 && k <= CSA2_MAX_TOPK, CSA2_ERR_RANGE, "k %d", k);
  const PrefillLayout L = prefill_layout(Q, cache->capacity, n_heads, k, cache->swa_dtype);
  const size_t need = csa2_prefill_workspace_size(Q, cache->capacity, n_heads_idx, n_heads, k);
  REQUIRE(ws != nullptr && ws_bytes >= need, CSA2_ERR_WORKSPACE, "prefill workspace %zu < %zu bytes", ws_bytes,
          need);
  REQUIRE(aligned16(ws), CSA2_ERR_ALIGN, "ws is not 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *wb = static_cast<uint8_t *>(ws);
  int64_t *P = reinterpret_cast<int64_t *>(wb + L.off_P);
  int64_t *qpos = reinterpret_cast<int64_t *>(wb + L.off_qpos);
  uint8_t *ring_c = wb + L.off_ring_c, *ring_s = wb + L.off_ring_s;
  uint8_t *lin_c = wb + L.off_lin_c, *lin_s = wb + L.off_lin_s;
  float *scores = reinterpret_cast<float *>(wb + L.off_scores);
  const csa2_cache v = seq_view(*cache, seq);

  g_phase_used = 0;
  mark_phase(s);  // start
  csa2::k_prefill_snapshot<<<64, 256, 0, s>>>(v, Q, P, qpos, ring_c, ring_s);
  cudaError_t e = csa2::launch_kv_append(v, nullptr, nullptr, CSA2_IN_F32, cmp, rope_cs, rope_len, Q, nullptr,
                                         err_word, s);
  if (e != cudaSuccess) return cuda_status(e, "prefill append");
  csa2::k_prefill_window<<<(Q + 7) / 8, 256, 0, s>>>(cmp->ca, Q, P, rope_cs, rope_len, cache->swa_dtype, lin_c,
                                                      cache->swa_dtype == CSA2_SWA_MXFP8 ? lin_s : nullptr);
  mark_phase(s);  // append and window rows done
  for (int q0 = 0; q0 < Q; q0 += L.qb) {
    const int nq = Q - q0 < L.qb ? Q - q0 : L.qb;
    csa2::ScoreArgs sa{};
    sa.idx_codes = v.idx_codes;
    sa.idx_scales = v.idx_scales;
    sa.map = csa2::entry_map(v);
    sa.cap = cache->capacity;
    sa.ratio = 2;
    sa.rows = nq;
    sa.heads = n_heads_idx;
    sa.q_idx = q_idx + static_cast<size_t>(q0) * n_heads_idx * csa2::kDi;
    sa.w = w + static_cast<size_t>(q0) * n_heads_idx;
    sa.q_pos = qpos + q0;
    sa.cache_seq = 0;
    sa.pool = nullptr;
    sa.scores = scores;
    sa.stride = cache->capacity;
    sa.aux = wb + L.off_aux;
    sa.err = err_word;
    sa.no_block_max = 1;  // the prefill's top-k builds no pool: the score histogram is all it reads
    e = csa2::launch_index_score_tc(sa, wb + L.off_qrec, s);
    if (e != cudaSuccess) return cuda_status(e, "prefill score");
    mark_phase(s);  // block scored
    csa2::TopkArgs se{};
    se.rows = nq;
    se.scores = scores;
    se.stride = cache->capacity;
    se.aux = wb + L.off_aux;
    se.ratio = 2;
    se.q_pos = qpos + q0;
    se.pool = nullptr;
    se.bs = 8;
    se.k = k;
    se.idx_out = idx_out + static_cast<size_t>(q0) * k;
    se.out_pool_blocks = 0;
    se.err = err_word;
    e = csa2::launch_topk(se, wb + L.off_sel, s);
    if (e != cudaSuccess) return cuda_status(e, "prefill top-k");
    mark_phase(s);  // block selected
    csa2::AttnArgs aa{};
    aa.rows = nq;
    aa.heads = n_heads;
    aa.k = k;
    aa.q = q + static_cast<size_t>(q0) * n_heads * csa2::kDqk;
    aa.idx = idx_out + static_cast<size_t>(q0) * k;
    aa.q_pos = qpos + q0;
    aa.cache_seq = 0;
    aa.lat_codes = v.lat_codes;
    aa.lat_scales = v.lat_scales;
    aa.rope_codes = v.rope_codes;
    aa.rope_scales = v.rope_scales;
    aa.map = csa2::entry_map(v);
    aa.entry_format = cache->entry_format;
    aa.cap = cache->capacity;
    aa.ratio = 2;
    aa.n_tokens = v.n_tokens;
    aa.ring_codes = ring_c;
    aa.ring_scales = cache->swa_dtype == CSA2_SWA_MXFP8 ? ring_s : nullptr;
    aa.ring_single = 1;
    aa.swa_dtype = cache->swa_dtype;
    aa.lin_codes = lin_c;
    aa.lin_scales = cache->swa_dtype == CSA2_SWA_MXFP8 ? lin_s : nullptr;
    aa.lin_base = P;
    aa.sink = sink;
    aa.sm_scale = sm_scale;
    aa.out = out + static_cast<size_t>(q0) * n_heads * csa2::kLat;
    aa.lse = lse + static_cast<size_t>(q0) * n_heads;
    aa.err = err_word;
    // one segment per query: each query's attention is one pass over its entries
    e = csa2::launch_attn(aa, 1, wb + L.off_attn, L.total - L.off_attn, s);
    if (e != cudaSuccess) return cuda_status(e, "prefill attention");
    mark_phase(s);  // block attended
  }
  return cuda_status(cudaGetLastError(), "csa2_prefill_chunk");
}

}  // extern "C"
