/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DSA sparse-attention step.
 *
 * The step (DeepSeek-V3.2-style DSA as used by GLM-5.2 decode and MTP verify):
 *   1. lightning indexer   I[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . k[s,:])
 *      over every cached index key s <= pos(t) of the query's request
 *      (mlx-lm "GLM-5.2 (glm_moe_dsa) inference", IndexShare commit, names the
 *      lightning indexer; lmdeploy "feat: support GLM-5.2", Changes: "DSA indexing");
 *   2. radix top-k         the index_topk largest I[t,s], ties to the lower s,
 *      ascending, -1 padded when fewer keys are causally valid
 *      (lmdeploy "feat: support GLM-5.2", Changes: radix top-k; lmdeploy
 *      "glm5.3-flash support", Operator-level gains: negative-index padding;
 *      mlx-lm small-L gather commit: re-masking when fewer than K keys are valid);
 *   3. sparse absorbed MLA over the selected 576-wide latent rows (512 latent +
 *      64 RoPE), value = the 512 latent columns, read straight from the paged
 *      cache (lmdeploy "feat: support GLM-5.2", Five-layer ablations: zero-copy
 *      BF16 sparse MLA; FP8 sparse FlashMLA cache path);
 *   IndexShare: a shared layer reuses the previous full layer's selection and
 *      skips steps 1-2 (mlx-lm IndexShare commit; lmdeploy shared top-k reuse).
 *
 * Conventions common to every entry point
 *   - Pointers named "device" must be device memory of the current CUDA device;
 *     the library never dereferences them on the host. All device buffers are
 *     owned by the caller; the library allocates no device memory, keeps no
 *     device state, and never synchronizes except in dsa_get_error().
 *   - `stream` is a cudaStream_t passed as void*; all work is enqueued on it.
 *   - Paged caches hold 64-token pages; page p holds tokens p*64 .. p*64+63 of
 *     whatever request maps it. Request b's logical token s lives in page
 *     block_table[b*bt_stride + s/64], row s%64.
 *   - Query positions: query j (0-based) of request b sits at position
 *     pos = seq_lens[b] - n_b + j with n_b = cu_q[b+1]-cu_q[b]; seq_lens counts
 *     the cached tokens including the query tokens' own keys. Keys 0..pos are
 *     visible to it.
 *   - Workspace: every compute entry point takes `ws`/`ws_bytes`, device memory
 *     of at least the size its *_workspace_size() function returns (256 bytes for
 *     dsa_wait_probe; dsa_stage_copy takes none), 256-byte aligned.
 *     Its first 256 bytes hold the device error word; zero them once before
 *     first use (dsa_clear_error). Calls on the same workspace must be ordered
 *     on one stream. The header's second int32 counts the score segments (rows,
 *     or 16384-position chunks of longer rows) whose first-digit histogram the
 *     step's top-k found not to match the scores (dsa_decode_step_hist, below); it
 *     is diagnostic only and dsa_clear_error zeroes it.
 *   - Host-side argument errors return DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED
 *     / DSA_ERR_WORKSPACE before anything is enqueued. Zero work (T == 0) is a
 *     no-op returning DSA_OK. Launch failures return DSA_ERR_CUDA.
 *   - Device-side data errors (a page id outside [0, num_pages), seq_lens or
 *     cu_q inconsistent with the host sizes, a selected index outside the
 *     request) never fault: the offending element is skipped and the error word
 *     is set to DSA_ERR_BAD_INDEX; a bounded wait that expires sets
 *     DSA_ERR_TIMEOUT. dsa_get_error() reports either.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 1

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,
  DSA_ERR_UNSUPPORTED = 2,
  DSA_ERR_CUDA = 3,
  DSA_ERR_TIMEOUT = 4,
  DSA_ERR_WORKSPACE = 5,
  DSA_ERR_BAD_INDEX = 6
} dsa_status_t;

typedef enum { DSA_BF16 = 0, DSA_E4M3 = 1, DSA_I8 = 2 } dsa_dtype_t;

/* Request geometry shared by every entry point. */
typedef struct {
  int32_t B;                  /* requests, >= 0 (no upper bound)                     */
  int32_t T;                  /* flattened query tokens = cu_q[B], >= 0              */
  int32_t max_seq_len;        /* host upper bound on every seq_lens[b], >= 1; sizes the
                                 grids and the top-k levels                          */
  int32_t num_pages;          /* physical pages in each paged cache, 1 .. 2^31/64    */
  int32_t page_size;          /* must be 64                                          */
  int32_t bt_stride;          /* int32 elements between block-table rows,
                                 >= ceil(max_seq_len/64)                             */
  const int32_t* seq_lens;    /* device [B]    cached tokens incl. the query tokens  */
  const int32_t* cu_q;        /* device [B+1]  query-token offsets, cu_q[0] = 0      */
  const int32_t* block_table; /* device [B, bt_stride] physical page ids             */
} dsa_geom_t;

/*
 * dsa_indexer_scores -- step 1 (lightning indexer).
 *   qk_dtype DSA_E4M3: q_idx [T, Hi, 128] e4m3 bytes, q_scale [T, Hi] fp32,
 *     idx_k_cache [num_pages, 64, 128] e4m3 bytes, idx_k_scale [num_pages, 64] fp32
 *     (one scale per token); the scores use q = code*q_scale, k = code*k_scale.
 *   qk_dtype DSA_BF16: q_idx [T, Hi, 128] bf16, idx_k_cache [num_pages, 64, 128]
 *     bf16; q_scale and idx_k_scale must be NULL.
 *   w [T, Hi] fp32 head weights. 1 <= Hi <= 64; the kernel pads the heads to 16 or 64
 *     with zero weights (when Hi is a multiple of 4 the w and q_scale rows move as
 *     16-byte bulk copies, otherwise 4 bytes at a time). Any B: requests are scored in
 *     launches of up to 1024 each.
 *   scores [T, score_stride] fp32 (device, written): for query t and s <= pos(t),
 *     scores[t*score_stride + s] = I[t,s]; entries pos(t) < s < seq_len are set to
 *     -inf; entries s >= seq_len are not written. score_stride >= max_seq_len.
 *   All pointers device, 16-byte aligned; tensors are contiguous.
 */
dsa_status_t dsa_indexer_scores(const dsa_geom_t* geom, dsa_dtype_t qk_dtype, int32_t Hi,
                                const void* q_idx, const float* q_scale, const float* w,
                                const void* idx_k_cache, const float* idx_k_scale,
                                float* scores, int64_t score_stride,
                                void* ws, size_t ws_bytes, void* stream);
size_t dsa_indexer_scores_workspace_size(const dsa_geom_t* geom);

/*
 * dsa_topk -- step 2 (radix top-k), exact.
 *   scores [T, score_stride] fp32 (device, read): row t is read at s = 0..pos(t) only.
 *   idx [T, k] int32 (device, written): the min(k, pos(t)+1) positions with the
 *     largest scores, ties broken toward the lower position, in ascending order,
 *     followed by -1 up to k. -0.0 and +0.0 compare equal. Scores must not be NaN.
 *   1 <= k <= 16384. Rows of up to 16384 positions are selected in one pass; longer
 *     rows are cut into 16384-position chunks whose top-k lists (keys and positions, in
 *     the workspace) are merged min(4, floor(16384/k)) at a time, level after level, so any
 *     max_seq_len works when k <= 8192; k > 8192 with max_seq_len > 16384 returns
 *     DSA_ERR_UNSUPPORTED.
 */
dsa_status_t dsa_topk(const dsa_geom_t* geom, const float* scores, int64_t score_stride,
                      int32_t k, int32_t* idx, void* ws, size_t ws_bytes, void* stream);
size_t dsa_topk_workspace_size(const dsa_geom_t* geom, int32_t k);

/*
 * dsa_sparse_mla_attend -- step 3 (absorbed MLA over the selected latent rows).
 *   q [T, H, 576] bf16 (device): the absorbed query (W_UK already folded in).
 *   kv_dtype DSA_BF16: kv_cache [num_pages, 64, 576] bf16.
 *   kv_dtype DSA_E4M3: kv_cache [num_pages, 41984] bytes, 656 per token: 512 e4m3
 *     latent codes, 4 little-endian fp32 scales (latent element 128c+e is
 *     code*scale[c]), 64 bf16 RoPE values. Each page holds its 64 tokens' fields as
 *     three planes: codes [64][512] at byte 0, scales [64][4] at byte 32768, RoPE
 *     [64][64] at byte 33792 (token s of the page: codes at 512*s, scales at
 *     32768 + 16*s, RoPE at 33792 + 128*s).
 *   kv_dtype DSA_I8: the same record pages with two's-complement int8 codes
 *     (the int8 latent cache of mlx-lm "GLM-5.2 (glm_moe_dsa) inference": only
 *     the compressed latent is quantized; dequantized on read).
 *   idx [T, k] int32 (device): logical positions of the request's tokens; -1 is
 *     padding and is skipped.
 *   For each (t, h): z_i = sm_scale * q[t,h,:] . kv[s_i,:] over the selected s_i,
 *     out[t,h,:] = sum_i softmax(z)_i * kv[s_i, 0:512]  (bf16, [T, H, 512])
 *     lse[t,h]   = ln(sum_i exp(z_i))                    (fp32, [T, H], or NULL)
 *   An all-padding row gives out = 0 and lse = -inf.
 *   out and lse: device memory, or page-locked host memory that the device maps
 *     (cudaHostAlloc, or cudaHostRegister with cudaHostRegisterMapped): the kernels
 *     then write the results straight to the host, and the stream's completion means
 *     they are there. Anything else (pageable host memory) is DSA_ERR_INVALID_ARG.
 *   H: 1..16 or a multiple of 16 up to 128. 1 <= k <= 16384.
 */
dsa_status_t dsa_sparse_mla_attend(const dsa_geom_t* geom, dsa_dtype_t kv_dtype, int32_t H,
                                   const void* q, const void* kv_cache, const int32_t* idx,
                                   int32_t k, float sm_scale, void* out, float* lse,
                                   void* ws, size_t ws_bytes, void* stream);
size_t dsa_sparse_mla_attend_workspace_size(const dsa_geom_t* geom, int32_t H, int32_t k);

/*
 * dsa_sparse_mla_attend_static -- dsa_sparse_mla_attend for callers that cannot
 *   provide device memory at call time: a runtime that plans and reserves all of
 *   its device memory up front, a plugin host that offers no workspace, or code
 *   at a point where an allocation would synchronize the device or disturb a
 *   memory pool. It takes no workspace and allocates nothing; the split-softmax
 *   partials live in a library-owned static device buffer of
 *   DSA_STATIC_SCRATCH_BYTES per GPU, which every GPU that loads the library
 *   holds until the process exits. (The pages have no counterpart to this entry
 *   point.)
 *   Arguments, layouts and results are those of dsa_sparse_mla_attend, except:
 *   err_word: device int32, 4-byte aligned, not NULL: it receives device-side data
 *     errors (DSA_ERR_BAD_INDEX, DSA_ERR_TIMEOUT); the caller zeroes it. (A bounded
 *     wait that gives up leaves the call's partial rows unwritten, and the merge would
 *     read an earlier call's; the error word is what reports it.)
 *   The call needs (T + G) * H * 2056 bytes of the buffer (G = min(SM count,
 *   T * ceil(k/128))); a larger call returns DSA_ERR_WORKSPACE and
 *   dsa_last_error() says how much was needed.
 *   The first call on a device looks up the buffer's address on that device;
 *   make that first call before any stream capture. Every call shares the buffer
 *   and it keeps the last call's contents (nothing in it must start at zero);
 *   calls whose work overlaps on the GPU race on it.
 */
#define DSA_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
dsa_status_t dsa_sparse_mla_attend_static(const dsa_geom_t* geom, dsa_dtype_t kv_dtype, int32_t H,
                                          const void* q, const void* kv_cache, const int32_t* idx,
                                          int32_t k, float sm_scale, void* out, float* lse,
                                          int32_t* err_word, void* stream);

/*
 * dsa_cache_append -- write the new tokens' latent rows and index keys into the
 *   paged caches (the cache update that runs before each decode / draft step's
 *   attention; lmdeploy "feat: support GLM-5.2", Changes: BF16/FP8 sparse
 *   FlashMLA cache paths, MLA cache dtype policy; lmdeploy "glm5.3-flash
 *   support": cache updates still run on every draft step).
 *   The new tokens are flattened like queries: token j of request b is the
 *     request's position seq_lens[b] - n_b + j (n_b from cu_q), written to page
 *     block_table[b][pos/64], row pos%64 -- the row the indexer and attention
 *     read for that position. geom->T is the number of new tokens.
 *   kv_new [T, 576] bf16 (device): latent (512) then RoPE (64) of each token.
 *   kv_dtype DSA_BF16: kv_cache [num_pages, 64, 576] bf16 receives kv_new as is.
 *   kv_dtype DSA_E4M3: kv_cache [num_pages, 41984] bytes (the record pages of
 *     dsa_sparse_mla_attend) receives, per token, for each group c of 128 latent
 *     values scale_c = amax_c / 448 (fp32; 1 for an all-zero group) and
 *     code = e4m3(x / scale_c) (quotient in fp32, round to nearest even, saturating
 *     at +-448): its 512 codes, 4 scales (little-endian fp32) and 64 RoPE values
 *     (bf16) at its slot of the page's three planes.
 *   kv_dtype DSA_I8: the same record with scale_c = amax_c / 127 and int8 codes
 *     round-to-nearest-even(x / scale_c) clamped to +-127.
 *   k_new [T, 128] bf16 (device) or NULL to leave the index cache alone.
 *   qk_dtype DSA_E4M3: idx_k_cache [num_pages, 64, 128] e4m3 and idx_k_scale
 *     [num_pages, 64] fp32 receive codes and one scale per token, same rule.
 *   qk_dtype DSA_BF16: idx_k_cache [num_pages, 64, 128] bf16 receives k_new as
 *     is; idx_k_scale must be NULL.
 *   No other row changes. All pointers 16-byte aligned. A page id out of range
 *   skips that token and sets DSA_ERR_BAD_INDEX in the error word.
 */
dsa_status_t dsa_cache_append(const dsa_geom_t* geom, dsa_dtype_t kv_dtype, const void* kv_new,
                              void* kv_cache, dsa_dtype_t qk_dtype, const void* k_new,
                              void* idx_k_cache, float* idx_k_scale, void* ws, size_t ws_bytes,
                              void* stream);
size_t dsa_cache_append_workspace_size(const dsa_geom_t* geom);

/*
 * dsa_indexer_prepare -- the indexer's query/key preparation, fused into one launch
 *   (lmdeploy "feat: support GLM-5.2", Changes: fused indexer preparation;
 *   mlx-lm "GLM-5.2 (glm_moe_dsa) inference", Changes: the indexer's RoPE is
 *   non-interleaved and its LayerNorm eps is 1e-6). It produces the e4m3 queries
 *   and scales dsa_indexer_scores takes, and writes each new token's key into the
 *   e4m3 index cache, for query token t (flattened like the queries) at position
 *   pos(t) = seq_lens[b] - n_b + j:
 *     q_out[t,h,:] = e4m3(RoPE(q_in[t,h,:]) / s), q_scale[t,h] = s
 *     idx_k_cache[row(pos(t)),:] = e4m3(RoPE(LayerNorm(k_in[t,:])) / s_k),
 *     idx_k_scale[row(pos(t))] = s_k
 *   RoPE (non-interleaved) on the first rope_dim values: for i < r = rope_dim/2,
 *     y_i = x_i*cos[pos][i] - x_{i+r}*sin[pos][i], y_{i+r} = x_{i+r}*cos[pos][i] +
 *     x_i*sin[pos][i]; values rope_dim..127 pass through.
 *   LayerNorm: (x - mean) / sqrt(var + ln_eps) * gamma + beta over the 128 values,
 *     var the biased variance; gamma NULL means 1, beta NULL means 0.
 *   s = amax / 448 of the vector (1 if it is all zero); codes round to nearest
 *   (ties to even) and saturate at +-448; everything is computed in fp32 from the
 *   bf16 inputs.
 *   Hi: 1..128 indexer heads. rope_dim: 8..128, a multiple of 8.
 *   q_in [T, Hi, 128] bf16, k_in [T, 128] bf16 or NULL (queries only; then the
 *     caches may be NULL); rope_cos, rope_sin [max_seq_len, rope_dim/2] fp32;
 *     ln_gamma, ln_beta [128] fp32 or NULL; q_out [T, Hi, 128] e4m3 bytes;
 *     q_scale [T, Hi] fp32; idx_k_cache [num_pages, 64, 128] e4m3 bytes;
 *     idx_k_scale [num_pages, 64] fp32. All device, 16-byte aligned (scales 4).
 *   Rows other than the new tokens' are untouched. A token whose page id is out
 *   of range is skipped and sets DSA_ERR_BAD_INDEX in the error word.
 */
dsa_status_t dsa_indexer_prepare(const dsa_geom_t* geom, int32_t Hi, int32_t rope_dim, const void* q_in,
                                 const void* k_in, const float* rope_cos, const float* rope_sin,
                                 const float* ln_gamma, const float* ln_beta, float ln_eps, void* q_out,
                                 float* q_scale, void* idx_k_cache, float* idx_k_scale, void* ws, size_t ws_bytes,
                                 void* stream);
size_t dsa_indexer_prepare_workspace_size(const dsa_geom_t* geom);

/*
 * dsa_stage_copy -- copies `bytes` from src to dst with the GPU's SMs, as a kernel in
 *   `stream`: for moving a step's packed inputs from page-locked host memory to the
 *   device and its outputs back. On a part whose host memory is reached over a
 *   coherent chip-to-chip link this beats a copy-engine transfer of the same size.
 *   Not part of the DSA method (the pages have no counterpart); the step's own
 *   entry points take device memory as before.
 *   Each range must lie in device (or managed) memory, or in page-locked host memory
 *   the device maps (cudaHostAlloc, cudaHostRegister), and be 16-byte aligned; both
 *   ends of each range are resolved with cudaPointerGetAttributes and must map
 *   contiguously, otherwise DSA_ERR_INVALID_ARG before anything is enqueued
 *   (pageable host memory is refused). The ranges must not overlap. bytes == 0 is a
 *   no-op.
 */
dsa_status_t dsa_stage_copy(void* dst, const void* src, size_t bytes, void* stream);

/* Arguments of the fused step. */
typedef struct {
  dsa_geom_t geom;
  int32_t topk;                /* index_topk, 1..16384                                  */
  /* indexer inputs (ignored when reuse_idx != NULL) */
  dsa_dtype_t qk_dtype;
  int32_t Hi;
  const void* q_idx;
  const float* q_scale;
  const float* w;
  const void* idx_k_cache;
  const float* idx_k_scale;
  /* IndexShare: a shared layer passes the full layer's selection here [T, topk] */
  const int32_t* reuse_idx;
  /* optional output of the selection [T, topk] (for the next shared layers) */
  int32_t* idx_out;
  /* attention inputs and outputs */
  dsa_dtype_t kv_dtype;
  int32_t H;
  const void* q;
  const void* kv_cache;
  float sm_scale;
  void* out;                   /* [T, H, 512] bf16; device or mapped page-locked host memory */
  float* lse;                  /* [T, H] fp32 or NULL; the same */
} dsa_step_args_t;

/*
 * dsa_decode_step -- the fused DSA step on one stream: indexer -> top-k ->
 *   sparse MLA (+ split combine), or, with reuse_idx != NULL (IndexShare), the
 *   sparse MLA alone over reuse_idx. No host synchronization; the enqueued work
 *   depends only on the host fields of `args`, so it can be captured in a CUDA
 *   graph. Scores and (when idx_out is NULL) the selection live in `ws`.
 */
dsa_status_t dsa_decode_step(const dsa_step_args_t* args, void* ws, size_t ws_bytes,
                             void* stream);
size_t dsa_decode_step_workspace_size(const dsa_step_args_t* args);

/*
 * dsa_decode_step_hist -- dsa_decode_step with the top-k's first radix digit
 *   counted by the indexer (the first pass of the radix top-k, lmdeploy "feat:
 *   support GLM-5.2", Changes, moved into the epilogue that makes the scores): per
 *   query and per 16384-position chunk of its row, the indexer counts the top 11 bits
 *   of every visible score's radix key in shared memory and adds them into histograms
 *   held in the last T * ceil(max(max_seq_len, 1) / 16384) * 8 KB of the
 *   workspace size this call asks for; the top-k reads them instead
 *   of counting the digit itself and leaves them zero for the next call. Each
 *   selection so made is checked against its exact final counts, so histograms that
 *   do not belong to the scores (a workspace's first use, or one that other calls
 *   wrote over) cost time, not exactness: the segment is selected again without them,
 *   and the header's second word counts it. Results are bitwise those of
 *   dsa_decode_step. With bf16 index keys (whose query-group variants leave the
 *   indexer no shared memory for the counts) the call runs as dsa_decode_step. On
 *   GB300 it is slower than dsa_decode_step (the counts cost the indexer more than
 *   they save the top-k), which stays the default.
 */
dsa_status_t dsa_decode_step_hist(const dsa_step_args_t* args, void* ws, size_t ws_bytes, void* stream);
size_t dsa_decode_step_hist_workspace_size(const dsa_step_args_t* args);

/*
 * dsa_decode_step_wait_q -- dsa_decode_step for a caller whose MLA query (args->q)
 *   may still be on its way to the device when the call is enqueued: the indexer
 *   and top-k are enqueued as usual, and the sparse-MLA attention waits on the CUDA
 *   event q_ready (cudaEvent_t, recorded after q's copy, e.g. on another stream)
 *   before it starts; NULL behaves as dsa_decode_step. Same results. (Not a step of
 *   the method: it lets the copy of the largest per-step input overlap the indexer.)
 */
dsa_status_t dsa_decode_step_wait_q(const dsa_step_args_t* args, void* q_ready, void* ws, size_t ws_bytes,
                                    void* stream);

/*
 * dsa_decode_step_bounded -- dsa_decode_step with the indexer's score workspace
 *   bounded (lmdeploy "glm5.3-flash support", Capacity improvement: bounded KPool
 *   scoring: a configurable score budget, top-k selected per query chunk right after
 *   that chunk is scored, indices identical). With R = (max_seq_len rounded up to 64)
 *   * 4 bytes, one query's score row:
 *   - budget >= R: the fp32 scores of floor(budget / R) queries exist at a time; each
 *     such range of queries is scored and reduced to its selection before the next.
 *   - 65536 <= budget < R: one query at a time, its keys in spans of
 *     floor(budget / 65536) * 16384 positions; each span is scored and reduced to the
 *     top-k lists of its 16384-position chunks before the next span, and the lists are
 *     merged at the end (as dsa_topk does for long rows), so the scores of at most
 *     one span exist at a time whatever the context length.
 *   - budget < min(R, 65536): DSA_ERR_INVALID_ARG (dsa_last_error gives the sizes).
 *   Results (idx_out, out, lse) are bitwise those of dsa_decode_step. With reuse_idx
 *   the budget is not used. Graph-capturable like dsa_decode_step.
 */
dsa_status_t dsa_decode_step_bounded(const dsa_step_args_t* args, size_t score_budget_bytes, void* ws,
                                     size_t ws_bytes, void* stream);
size_t dsa_decode_step_bounded_workspace_size(const dsa_step_args_t* args, size_t score_budget_bytes);

/* Synchronizes `stream`, reads the device error word of `ws` (DSA_OK if none)
 * and clears it. Returns DSA_ERR_CUDA if the stream itself reports an error. */
dsa_status_t dsa_get_error(void* ws, void* stream);
/* Enqueues a clear of the error word of `ws` on `stream`. */
dsa_status_t dsa_clear_error(void* ws, void* stream);

/*
 * dsa_wait_probe -- runs the failure path of the kernels' bounded waits on purpose.
 *   Every pipeline wait (an mbarrier phase completed by a copy, an MMA or another
 *   warp) gives up after a time limit and records DSA_ERR_TIMEOUT in the workspace's
 *   error word instead of hanging. This call enqueues one block whose thread waits
 *   on an mbarrier phase that nothing completes, for at most limit_us microseconds
 *   (1 .. 1,000,000), then records DSA_ERR_TIMEOUT in `ws`'s error word and exits.
 *   Read it with dsa_get_error; the context stays usable.
 *   ws: device, 256-byte aligned, ws_bytes >= 256. Returns DSA_ERR_INVALID_ARG for a
 *   limit out of range, DSA_ERR_WORKSPACE for a missing or misaligned workspace,
 *   DSA_ERR_CUDA if the launch fails.
 */
dsa_status_t dsa_wait_probe(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream);

const char* dsa_status_string(dsa_status_t status);
/* Text describing the last failure seen by an entry point on the calling host
 * thread (the failing call and its CUDA error), or "" if none. Owned by the
 * library; valid until the next entry-point call on the same thread. */
const char* dsa_last_error(void);
int32_t dsa_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H_ */
