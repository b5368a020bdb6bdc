/*
 * csa2.h -- C ABI of libcsa2, the CSA2 long-context attention step
 * (FP4 global KV cache, lightning indexer, top-k, sparse absorbed-query
 * attention with a sliding window) on one GB300 (sm_103a).
 *
 * Source pages cited below:
 *   [P1] "DeepSeek V4.1 Flash 아키텍처 분석" (plaidlabs.ai blog)
 *   [P2] "DeepSeek Multi-Head Latent Attention(MLA) 해부" (huny.dev blog)
 *   [P3] "DeepSeek V4.1 Flash 해부, KV 캐시는 줄고 사후학습 레시피는 그대로" (traillabs.ai)
 *   [P4] "매개변수는 커졌는데 메모리는 4분의 1, DeepSeek V4.1 Flash의 KV 캐시 다이어트" (ithotfix.com)
 *   [P5] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence" (issue #58 translation)
 *
 * Conventions (all calls):
 *   - The caller owns every buffer.  Device pointers are CUDA device memory of
 *     the current device; host pointers are marked (host).  The library never
 *     allocates on these calls; scratch comes from a caller workspace whose
 *     size the matching *_workspace_size() returns.
 *   - Every device pointer must be 16-byte aligned (CSA2_ERR_ALIGN otherwise).
 *   - Calls are asynchronous on the given stream (a cudaStream_t; NULL = the
 *     legacy default stream).  They validate their arguments on the host first
 *     and return a status; they never abort and never throw.
 *   - Errors that only the device can see (an append beyond the capacity, an
 *     index outside the cache, a NaN score) set bits of the caller's int32
 *     *err_word (device memory, may be NULL to ignore) with atomicOr; the
 *     affected outputs are then unspecified.  Clear it before the calls and
 *     read it after synchronising.
 *   - csa2_last_error_detail() returns a thread-local text for the last
 *     non-OK status of this thread.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *csa2_stream_t;

typedef enum csa2_status {
  CSA2_OK = 0,
  CSA2_ERR_NULL = 1,        /* a required pointer is NULL                       */
  CSA2_ERR_SHAPE = 2,       /* a size is outside its documented range           */
  CSA2_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned          */
  CSA2_ERR_RANGE = 4,       /* an enum / k / ratio argument is out of range      */
  CSA2_ERR_UNSUPPORTED = 5, /* valid but not implemented (e.g. ratio-1 prefill) */
  CSA2_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed      */
  CSA2_ERR_WORKSPACE = 7    /* the workspace is NULL or smaller than required   */
} csa2_status;

/* bits of the device error word */
#define CSA2_DEVERR_CAPACITY 1u /* append past the cache capacity (nothing written) */
#define CSA2_DEVERR_INDEX 2u    /* an index / pool id outside the visible cache (skipped) */
#define CSA2_DEVERR_NAN 4u      /* a NaN index score (it ranks lowest)                */
#define CSA2_DEVERR_ROPE 8u     /* a position outside the RoPE table (nothing written) */
#define CSA2_DEVERR_TIMEOUT 16u /* a bounded device wait gave up (outputs unspecified)  */
#define CSA2_DEVERR_INEXACT 32u /* an index score may not be the exact dot (see csa2_index_score) */

/* sliding-window storage */
#define CSA2_SWA_BF16 0  /* 576 bf16 values, 1,152 B per token                         */
#define CSA2_SWA_MXFP8 1 /* 576 E4M3 codes + 18 E8M0 scales (one per 32), 594 B/token */

/* main-entry formats of the global cache (csa2_cache.entry_format):
 *   CSA2_ENTRY_FP4: V4.1, the 288 B record: lat_codes 256 B (E2M1 x 512),
 *     lat_scales 32 B (E4M3 per 16); RoPE sidecar rope_codes 32 B, rope_scales 4 B.
 *   CSA2_ENTRY_FP8: V4 ([P5] §2.3.4: FP8 for the entry except the RoPE dims,
 *     which stay BF16), for comparison: lat_codes 512 B (E4M3 x 512), lat_scales
 *     16 B (one E8M0 per 32 latent dims, e = floor(log2 amax) - 8, as the 8-bit
 *     window), rope_codes 128 B (the 64 rotated RoPE dims in bf16), rope_scales
 *     unused (may be NULL): 656 B.  The indexer key is MXFP4 (68 B) in both. */
#define CSA2_ENTRY_FP4 0
#define CSA2_ENTRY_FP8 1

/* input element types for csa2_kv_append */
#define CSA2_IN_F32 0
#define CSA2_IN_BF16 1

/* Fixed dimensions of the path (see the citations on csa2_cache). */
#define CSA2_D_LATENT 512 /* latent dims of a main-KV entry ([P1] "890 bytes/token")       */
#define CSA2_D_ROPE 64    /* decoupled RoPE dims ([P2] §3; [P5] §2.3.3 "last 64 dims")     */
#define CSA2_D_QK 576     /* score dims of an absorbed query: latent + RoPE ([P2] §4)      */
#define CSA2_D_INDEX 128  /* indexer head dim c_I ([P5] §4.2.1)                            */
#define CSA2_D_CMP 704    /* one compression row: 576 main dims then 128 indexer dims      */
#define CSA2_WINDOW 128   /* sliding window n_win ([P5] §4.2.1)                            */
#define CSA2_MAX_TOPK 2048
#define CSA2_MAX_HEADS 128

/*
 * One global-KV cache (the output of one Full layer; Reindex and Reuse layers
 * read it).  Every plane is [batch][capacity][bytes], sequence-major, so one
 * sequence's entries are contiguous.  Per entry ([P1] "890 bytes/token";
 * [P4] "890이 맞아떨어지는 계산"):
 *   lat_codes   256 B  E2M1 codes of the 512 latent dims, byte j = code(2j) | code(2j+1) << 4
 *   lat_scales   32 B  one E4M3 scale per 16 dims                 -> 288 B main entry
 *   rope_codes   32 B  E2M1 codes of the 64 rotated RoPE dims (sidecar of the MLA split, [P2] §3)
 *   rope_scales   4 B  one E4M3 scale per 16                       -> 36 B sidecar
 *   idx_codes    64 B  E2M1 codes of the 128-dim indexer key
 *   idx_scales    4 B  one E8M0 scale per 32 (MXFP4)               -> 68 B indexer entry
 *   The two indexer planes are tile-major: [batch][ceil(capacity/128)][8192 B]
 *   and [batch][ceil(capacity/128)][512 B], in the operand layout of the
 *   block-scaled tensor-core MMA.  For entry e (tile = e/128, m = e%128) the
 *   16 code bytes of 32-value block j sit at tile*8192 + j*2048 + m*16 and its
 *   scale byte at tile*512 + 16*(m%32) + 4*(m/32) + j.  csa2_cache_plane_bytes()
 *   gives every plane's size.
 * swa_codes / swa_scales: the sliding-window ring, [batch][128][576] codes
 *   (E4M3 bytes, or bf16 when swa_dtype == CSA2_SWA_BF16) and [batch][128][32]
 *   scale bytes (18 used, MXFP8 only); token t lives in slot t % 128 ([P5]
 *   §3.5.1: the window is a fixed-size per-sequence state).
 * cmp_buf: ratio 2 only, float [batch][4][4][704]: the last tokens' compression
 *   rows (C^a, C^b, Z^a, Z^b) at slot t % 4, carried between appends ([P5] §3.5.1
 *   "Compression Buffer").
 * n_tokens: int64 [batch] tokens appended so far (device; csa2_kv_append and
 *   csa2_prefill_chunk advance it).  A ratio-r cache holds floor(n_tokens/r) entries.
 * ratio: 1 (one token per entry, decoder) or 2 (two tokens per entry, encoder;
 *   [P1] "Global KV는 네 곳에서 만든다", [P4] 178 B per token).
 *
 * Paged layout ([P5] §3.5.1 "Sparse Attention Kernel Co-Design": the global
 * entries live in fixed-size blocks whose token count is a multiple of the
 * compression ratios; the window and the compression buffer are
 * per-sequence state, "State Cache"): with block_table != NULL the six entry
 * planes hold n_pages physical pages of page_entries entries each, page-major
 * (lat_codes [n_pages][page_entries][256], ..., the indexer planes
 * [n_pages][page_entries/128][8192 B] and [..][512 B] in the same tile layout),
 * and entry e of sequence b is entry e % page_entries of physical page
 * block_table[b * max_pages + e / page_entries].  page_entries is a multiple of
 * 128 (an indexer tile never straddles pages; a page's tokens are then a
 * multiple of every ratio and of the 8-position pool block), capacity must
 * equal max_pages * page_entries, and page ids lie in 0..n_pages-1 (an id
 * outside raises the INDEX device bit and the access is skipped).  Pages may be
 * shared between sequences only for entries they hold in common; the caller
 * fills the table before the entries are appended.  The window ring, the
 * compression buffer and n_tokens stay indexed by sequence.  block_table ==
 * NULL: the dense layout above (page fields ignored).
 */
typedef struct csa2_cache {
  int32_t batch;
  int32_t capacity; /* entries per sequence */
  int32_t ratio;
  int32_t swa_dtype;
  uint8_t *lat_codes, *lat_scales;
  uint8_t *rope_codes, *rope_scales;
  uint8_t *idx_codes, *idx_scales;
  uint8_t *swa_codes, *swa_scales;
  float *cmp_buf;
  int64_t *n_tokens;
  const int32_t *block_table; /* [batch][max_pages] physical page ids, or NULL (dense) */
  int32_t page_entries;       /* entries per page: a multiple of 128 */
  int32_t max_pages;          /* pages a sequence may use: capacity / page_entries */
  int32_t n_pages;            /* physical pages in the entry planes */
  int32_t entry_format;       /* CSA2_ENTRY_FP4 (V4.1) or CSA2_ENTRY_FP8 (V4) */
} csa2_cache;

/* Ratio-2 compression inputs ([P5] §2.3.1 "압축된 Key-Value Entry"): per token
 * rows of C^a, C^b, Z^a, Z^b ([batch][n_new][704], device fp32) and the
 * positional biases B^a, B^b ([2][704], device fp32). */
typedef struct csa2_compress_in {
  const float *ca, *cb, *za, *zb;
  const float *ba, *bb;
} csa2_compress_in;

/* Bytes each plane of a cache needs (host helper; no device work). */
size_t csa2_cache_plane_bytes(int32_t batch, int32_t capacity, int32_t plane /* 0..9 as listed */,
                              int32_t swa_dtype);
/* Bytes of entry plane 0..5 in the paged layout (n_pages pages of page_entries). */
size_t csa2_paged_plane_bytes(int32_t n_pages, int32_t page_entries, int32_t plane);
/* Bytes one entry takes in plane 0..5 for an entry format (0 for an unknown
 * format or plane; the dense and paged plane sizes above are for
 * CSA2_ENTRY_FP4, scale them by this for CSA2_ENTRY_FP8). */
size_t csa2_entry_plane_bytes(int32_t entry_format, int32_t plane);

/*
 * csa2_rope_table (host): cos/sin table for the 64 RoPE dims, rope_cs[pos][i][2]
 * = (cos, sin)(pos * theta^(-2i/64)) for i < 32, evaluated in double and rounded
 * to fp32, positions 0..n_pos-1 ([P5] §2.3.3 "Partial Rotary Positional
 * Embedding"; pairs (2i, 2i+1) interleaved).  out_host holds n_pos*64 floats.
 */
csa2_status csa2_rope_table(double theta, int64_t n_pos, float *out_host);

/*
 * csa2_kv_append: quantise n_new new tokens of every sequence into the cache,
 * at positions n_tokens[b] .. n_tokens[b]+n_new-1, then advance n_tokens.
 *   ratio 1: kv [batch][n_new][576] (512 latent, 64 RoPE dims not yet rotated),
 *            idx_key [batch][n_new][128], element type in_dtype; cmp = NULL.
 *            Entry t = token t: RoPE at position t, then quantise ([P4]
 *            "890이 맞아떨어지는 계산": quantisation after RoPE).
 *   ratio 2: cmp != NULL, kv = idx_key = NULL.  Entry i is emitted when tokens
 *            2i, 2i+1 are present: per channel a softmax over the 4 rows
 *            [Z^a_2i + B^a_0, Z^a_2i+1 + B^a_1, Z^b_2i-2 + B^b_0, Z^b_2i-1 + B^b_1]
 *            and the gated sum of the matching C rows ([P5] §2.3.1), computed in
 *            fp64 and rounded to fp32, then RoPE at position 2i, then quantised.
 *            Rows of earlier appends come from cmp_buf.
 *   Window: each of the last min(n_new, 128) tokens fills slot t % 128 with its
 *            own vector (ratio 1: kv; ratio 2: C^a[0:576]) rotated at t, in 8 bits
 *            or bf16 ([P1] "890 bytes/token": the window KV stays in FP8).
 * rope_cs: device table from csa2_rope_table with rope_len positions.
 * cmp_dbg: NULL, or device fp32 [batch][n_new/2+1][704] receiving each emitted
 *   ratio-2 entry before RoPE (row e = the e-th entry emitted by this call).
 * Device errors: CAPACITY (a sequence would exceed capacity; nothing written
 *   for it), ROPE (a position >= rope_len).
 */
csa2_status csa2_kv_append(const csa2_cache *cache, const void *kv, const void *idx_key,
                           int32_t in_dtype, const csa2_compress_in *cmp, const float *rope_cs,
                           int64_t rope_len, int32_t n_new, float *cmp_dbg, int32_t *err_word,
                           csa2_stream_t stream);

/*
 * csa2_index_score: lightning-indexer scores ([P5] §2.3.1, "I_{t,s} = sum_h
 * w_{t,h} ReLU(q_{t,h} . K_s)"), with the query quantised to MXFP4 like the
 * keys (the indexer QK product runs in FP4, [P5] §2.3.4).
 *   q_idx: bf16 [batch][n_heads_idx][128]; w: fp32 [batch][n_heads_idx];
 *   q_pos: int64 [batch] query positions; entry s is visible iff
 *          s < floor(q_pos / ratio) ([P5] §2.3.1).
 *   d_h is the dot of the dequantised vectors, rounded once to fp32.  That holds
 *   when the block exponents e_q,j + e_k,j of a (head, key) pair span at most 9
 *   binades over the blocks whose two scale codes are nonzero (always the case
 *   for N(0,1)-like data); a visible key whose pair with some head spans more
 *   raises the INEXACT bit (its scores are then unspecified in the last bits);
 *   score = fma chain over heads in order: acc = fma(w_h, max(d_h, +0), acc).
 * FULL (pool == NULL): scores[b][s] for every visible s (others untouched).
 * POOL (Reindex, [P1] "512개를 고르기 위해 ..."): pool [batch][pool_blocks] int32
 *   ascending block ids (-1 = empty); scores[b][j*pool_block_size + i] is the
 *   score of position pool[b][j]*pool_block_size + i when it is visible.
 * score_stride: floats per sequence in scores (>= capacity for FULL,
 *   >= pool_blocks*pool_block_size for POOL).  n_heads_idx in 1..128.
 * score_aux: NULL, or a device buffer of csa2_score_aux_size(batch,
 *   score_stride) bytes that receives a sideband for csa2_topk: per row a
 *   histogram of the scores' top 13 order bits and, in FULL mode, the max of
 *   every 8-position block with its histogram.  Owned by the caller; valid
 *   until the scores change.  Building it here costs no extra pass over them.
 * ws: device workspace of csa2_index_score_workspace_size() bytes (the
 *   quantised queries in the tensor-core operand layout).
 * The contraction runs on the tensor cores (block-scaled MXFP4 MMA) for FULL
 * and for POOL with pool_block_size 8; other block sizes use CUDA cores (the
 * sideband is then built by a second kernel over the scores).
 */
size_t csa2_index_score_workspace_size(int32_t batch, int32_t n_heads_idx);
size_t csa2_score_aux_size(int32_t batch, int64_t score_stride);
csa2_status csa2_index_score(const csa2_cache *cache, const uint16_t *q_idx, const float *w,
                             int32_t n_heads_idx, const int64_t *q_pos, const int32_t *pool,
                             int32_t pool_blocks, int32_t pool_block_size, float *scores,
                             int64_t score_stride, void *score_aux, void *ws, size_t ws_bytes,
                             int32_t *err_word, csa2_stream_t stream);

/*
 * csa2_topk: top-k selector ([P5] §2.3.1 "Top-k(I_{t,:})") over the candidates
 * csa2_index_score scored (same ratio / q_pos / pool arguments), ordered by
 * score descending then position ascending (ties go to the lower position;
 * -0 == +0; NaN ranks lowest and raises the NAN bit).  idx_out [batch][k]
 * receives the chosen positions in ascending order, padded with -1.
 * k in 1..2048.
 * score_aux: the sideband csa2_index_score wrote for these scores, or NULL
 *   (it is then rebuilt from the scores inside ws, one more pass over them).
 * FULL mode only: when pool_out != NULL also builds the candidate pool of the
 * Hierarchical Sparse Indexer ([P1], [P4]): positions are grouped in aligned
 * blocks of pool_block_size = 8, a block's score is the max over its visible
 * positions, and the top out_pool_blocks (1..2048) blocks by (max desc, block
 * asc) are written ascending to pool_out [batch][out_pool_blocks] (padded with
 * -1), with their number in pool_count [batch].
 * ws: device workspace of csa2_topk_workspace_size() bytes (enough with or
 *   without score_aux).
 * The selection is exact for any input; rows whose k-th score falls in a bin
 * holding more than 4096 scores take a slower exact path.
 */
size_t csa2_topk_workspace_size(int32_t batch, int64_t score_stride, int32_t k,
                                int32_t out_pool_blocks);
csa2_status csa2_topk(const float *scores, int64_t score_stride, const void *score_aux,
                      int32_t batch, int32_t ratio, const int64_t *q_pos, const int32_t *pool,
                      int32_t pool_blocks, int32_t pool_block_size, int32_t k, int32_t *idx_out,
                      int32_t out_pool_blocks, int32_t *pool_out, int32_t *pool_count, void *ws,
                      size_t ws_bytes, int32_t *err_word, csa2_stream_t stream);

/*
 * csa2_topk_noalloc: csa2_topk without a caller workspace, for callers that
 * may not allocate device memory while they run (a host framework that owns all
 * device allocations, a service whose memory budget is fixed at start-up, code
 * that must not hit the allocator's implicit synchronisation).  The source pages
 * have no counterpart: this is a library convenience, not a step of the method.
 * Same arguments and results as csa2_topk minus score_aux, ws and ws_bytes (the
 * sideband is always rebuilt from the scores).  Its scratch is a 4 MiB array
 * compiled into the library, resident on every GPU that loads it until the
 * process exits; calls needing more (csa2_topk_workspace_size() > 4 MiB, i.e.
 * large batch x score_stride) return CSA2_ERR_WORKSPACE with the sizes in
 * csa2_last_error_detail().  The first call on each device looks up the
 * array's device address (a runtime query), so make that first call before any
 * stream capture; the address is kept for the process, so a cudaDeviceReset
 * after that first call is not supported.  Every call shares the array and leaves its contents behind
 * (each call clears and rewrites what it reads): calls whose kernels may
 * overlap on the GPU -- different streams without ordering -- race.
 */
csa2_status csa2_topk_noalloc(const float *scores, int64_t score_stride, int32_t batch, int32_t ratio,
                              const int64_t *q_pos, const int32_t *pool, int32_t pool_blocks,
                              int32_t pool_block_size, int32_t k, int32_t *idx_out,
                              int32_t out_pool_blocks, int32_t *pool_out, int32_t *pool_count,
                              int32_t *err_word, csa2_stream_t stream);

/*
 * csa2_mask_to_pool: the Reindex selection in the form of the published
 * reference code ([P1] "DeepSeek V4.1 Flash 아키텍처 분석", §"공개 코드를 읽어 보니
 * 남는 차이": Indexer.forward scores every key, then masks the positions outside
 * the candidates), kept for comparison with scoring only inside the pool.
 * scores [batch][score_stride] FULL-mode scores (csa2_index_score with pool ==
 * NULL); every visible position s < floor(q_pos[b] / ratio) whose block
 * s / pool_block_size is not among pool[b] (ascending block ids, -1 padded,
 * pool_blocks per row) is set to -inf in place.  csa2_topk (FULL, k) over the
 * masked row then selects what csa2_topk over the pool's scores selects
 * whenever the pool holds at least k visible positions.  pool_block_size 1..64.
 */
csa2_status csa2_mask_to_pool(float *scores, int64_t score_stride, int32_t batch, int32_t ratio,
                              const int64_t *q_pos, const int32_t *pool, int32_t pool_blocks,
                              int32_t pool_block_size, csa2_stream_t stream);

/*
 * csa2_sparse_attn_decode: core attention of one decode step over the k
 * selected entries and the window ([P5] §2.3.1 "Shared Key-Value MQA": each
 * entry is key and value; [P2] §4 absorbed query: logits over 576 dims, values
 * the 512 latent dims; [P5] §2.3.3 window branch and attention sink).
 *   q: bf16 [batch][n_heads][576] (latent 512 then rotated RoPE 64);
 *   idx: int32 [batch][k] positions (-1 = empty) -- a Reuse layer passes its
 *        leader's list and cache ([P3] "CSA2의 세 가지 모드");
 *   window: tokens max(0, q_pos-127) .. q_pos that are < n_tokens[b];
 *   sink: fp32 [n_heads] or NULL; sm_scale: logit scale.
 *   z_j = sm_scale * q . e_j; p_j = exp(z_j - M) / (sum_j exp(z_j - M) + exp(sink_h - M));
 *   out: fp32 [batch][n_heads][512] = sum_j p_j c_j; lse: fp32 [batch][n_heads]
 *   = M + log(denominator) (-inf when there is nothing to attend to).
 * n_heads: a multiple of 16, 16..128.  k: 1..2048.
 * Batch invariance ([P5] §3.3): a row's result is bit-identical whatever the
 *   batch it is computed in.  Its 32-entry chunks (the k selected entries, then
 *   the window) are dealt to S = min(4, chunks) segments, S a function of k
 *   alone; each segment runs its own online softmax and the row merges the S
 *   partials in segment order.  Only the launch shape follows the batch and
 *   the GPU's SM count: how many CTAs share a row's segments, and how many
 *   heads (64, 32 or 16) a CTA takes.
 * ws: device workspace of csa2_attn_workspace_size() bytes, 16-byte aligned:
 *   the partial (O, m, l) of each segment of a row (S x 131 KB per row and
 *   64 heads), written and read within the call; calls that may run
 *   concurrently need separate workspaces.
 * Device errors: INDEX (an index >= the visible entries; that entry is skipped).
 */
size_t csa2_attn_workspace_size(int32_t batch, int32_t n_heads, int32_t k);
csa2_status csa2_sparse_attn_decode(const csa2_cache *cache, const uint16_t *q, int32_t n_heads,
                                    const int64_t *q_pos, const int32_t *idx, int32_t k,
                                    const float *sink, float sm_scale, float *out, float *lse,
                                    void *ws, size_t ws_bytes, int32_t *err_word,
                                    csa2_stream_t stream);

/*
 * csa2_prefill_chunk: encoder-style chunked prefill of sequence `seq` of a
 * ratio-2 cache.  Appends the Q tokens (as csa2_kv_append, ratio 2), then for
 * every query i (position P+i, P = n_tokens[seq] before the call): scores all
 * visible entries s < floor((P+i)/2) with its own indexer query (a dense FP4
 * contraction), keeps its top k, and attends over them plus its window tokens
 * max(0, P+i-127) .. P+i ([P5] §2.3.1, §2.3.3).
 *   cmp: rows [Q][704] for this sequence; q_idx bf16 [Q][n_heads_idx][128];
 *   w fp32 [Q][n_heads_idx]; q bf16 [Q][n_heads][576];
 *   idx_out int32 [Q][k]; out fp32 [Q][n_heads][512]; lse fp32 [Q][n_heads].
 * ws: device workspace of csa2_prefill_workspace_size() bytes (queries are
 *   scored, selected and attended in blocks: the block holds ~256 MB of fp32
 *   score rows, rounded down to a multiple of twice the current device's SM
 *   count, so the size depends on the device the call runs on; query it with
 *   that device current).
 * Each query's attention is one pass over its entries (one segment), so its
 * bits do not depend on the chunk's size either; they may differ in the last
 * bits from a decode step at the same position (csa2_sparse_attn_decode merges
 * S segments), within the attention tolerance.
 * Ratio-1 caches return CSA2_ERR_UNSUPPORTED.
 */
size_t csa2_prefill_workspace_size(int32_t Q, int32_t capacity, int32_t n_heads_idx,
                                   int32_t n_heads, int32_t k);
csa2_status csa2_prefill_chunk(const csa2_cache *cache, int32_t seq, const csa2_compress_in *cmp,
                               const float *rope_cs, int64_t rope_len, int32_t Q,
                               const uint16_t *q_idx, const float *w, int32_t n_heads_idx,
                               const uint16_t *q, int32_t n_heads, int32_t k, const float *sink,
                               float sm_scale, int32_t *idx_out, float *out, float *lse, void *ws,
                               size_t ws_bytes, int32_t *err_word, csa2_stream_t stream);

/*
 * csa2_mxf4_peak_launch: measurement helper (not a step of the method).
 * Launches n_ctas CTAs that each issue `iters` back-to-back block-scaled FP4
 * tensor-core MMAs (tcgen05 kind::mxf4, M 128 x N 128 x K 64, the index score's
 * instruction) on operands resident in shared memory: n_ctas x iters x
 * 2,097,152 FLOP.  The caller times it (events on `stream`) to get the dense
 * FP4 rate the prefill indexer's tensor-pipe utilisation is reported against
 * ([P5] §2.3.4: the indexer QK product runs in FP4).  sink: NULL, or device
 * uint32 [n_ctas] receiving one accumulator word per CTA.  err_word: the
 * TIMEOUT bit if the final wait gave up.  n_ctas 1..4096, iters 2..2^24.
 */
csa2_status csa2_mxf4_peak_launch(int32_t n_ctas, int32_t iters, uint32_t *sink, int32_t *err_word,
                                  csa2_stream_t stream);

/*
 * csa2_bounded_wait_check: self-check of the failure path (not a step of the
 * method).  Every wait inside the library's kernels is bounded: a wait that
 * runs out sets CSA2_DEVERR_TIMEOUT in the call's error word, the kernel frees
 * its tensor memory and returns, and the context stays usable.  This launches
 * one warp that holds 32 TMEM columns across the same bounded wait on an
 * mbarrier that one arrival completes (complete = 1: the wait succeeds, no bit
 * is set) or that nothing completes (complete = 0: the wait gives up after
 * `iters` polls of at most ~1 ms each and sets the TIMEOUT bit), so that a host
 * can see the bit arrive and keep using the device.  iters 1..64; err_word:
 * device int32, 4-byte aligned, required (OR-ed into, never cleared).
 * Asynchronous on `stream` like every other call.
 */
csa2_status csa2_bounded_wait_check(int32_t iters, int32_t complete, int32_t *err_word, csa2_stream_t stream);

/*
 * csa2_set_phase_events: measurement helper.  events: n_events cudaEvent_t
 * (created by the caller, owned by it) that this thread's next
 * csa2_prefill_chunk calls record on their stream, in order, at the phase
 * boundaries: the start, append + window rows done, then per block of queries
 * scored, selected, attended (each call restarts at the first event; events
 * beyond n_events are not recorded).  NULL / 0 stops the recording.
 * csa2_phase_events_recorded() gives how many the last call recorded.
 */
csa2_status csa2_set_phase_events(void *const *events, int32_t n_events);
int32_t csa2_phase_events_recorded(void);

/* Status text, and the thread-local detail of this thread's last failure. */
const char *csa2_status_string(csa2_status status);
const char *csa2_last_error_detail(void);
/* Library version, major*10000 + minor*100 + patch. */
int32_t csa2_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
