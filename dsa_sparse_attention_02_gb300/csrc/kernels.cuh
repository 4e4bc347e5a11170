// Internal interface between the host API layer and the kernel files.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include "common.cuh"
#include "dsa.h"

namespace dsa {

// ---- lightning indexer (indexer.cu)
struct IndexerArgs {
  GeomDev g;
  int Hi;
  const float* q_scale;   // [T, Hi] or null (bf16)
  const float* w;         // [T, Hi]
  const float* k_scale;   // [P*64] or null (bf16)
  float* scores;        // column s - key_begin of row t holds I[t, s]
  int64_t stride;
  int key_begin;        // keys [key_begin, key_end) are scored; key_begin a multiple of 128
  int key_end;          // a multiple of 128, or past every request's length
  bool q_group_box;     // map_q's box is a whole query group (indexer_q_box_rows): one copy per group
  int* hist;            // or null: first-digit histograms [T][hist_chunks][kHistBins] of the visible
  int hist_chunks;      //   scores, added to (the top-k reads them and leaves them zero); key_begin 0
  int* err;
};
// Rows of the query tensor map's box: a whole group of 4 queries when several queries
// share a unit and Hi fills the padded head count (16 or 64), else one query's Hi rows.
int indexer_q_box_rows(int Hi, bool multi_query);
// pdl: launched with programmatic stream serialization (the kernel reads only call
// inputs before its grid-dependency wait; the scores are written after it).
cudaError_t indexer_launch(bool fp8, int Hi, bool multi_query, const CUtensorMap& mk, const CUtensorMap& mq,
                           const IndexerArgs& A, int grid, bool pdl, cudaStream_t st);
int indexer_max_requests();   // requests per launch (a call with more loops over groups)
// Whether the indexer variant for these keys and heads counts first-digit histograms
// (IndexerArgs::hist); where it does not, the top-k must count the digit itself.
bool indexer_counts_hist(bool fp8, int Hi, bool multi_query);

// ---- radix top-k (topk.cu)
// Rows longer than topk_chunk_len() are cut into chunks of that length whose top-k
// lists are merged topk_fan_in(k) at a time over topk_merge_levels() levels (-1: k
// too large for rows that long).
int topk_chunk_len();
int topk_fan_in(int k);
int topk_merge_levels(int max_seq_len, int k);
size_t topk_workspace_bytes(int T, int max_seq_len, int k);
// pdl: the launch may overlap the tail of the kernel just before it on the stream
// (programmatic dependent launch); set only when that kernel is one of this library's
// and the geometry was complete before it started.
// hist: null, or the first-digit histograms the indexer counted for these scores,
// [T][chunks per row][kHistBins] ints (topk_hist_bytes); each CTA reads its row's (or
// chunk's) and zeroes it. A histogram that does not match the scores (a workspace's
// first use) is detected by the selection's exact final counts, and the row is then
// selected without it.
cudaError_t topk_launch(const GeomDev& g, const float* scores, int64_t stride, int k, int* idx,
                        void* scratch, int* err, bool pdl, cudaStream_t st, int* hist = nullptr);
size_t topk_hist_bytes(int T, int max_seq_len);
int topk_row_chunks(int max_seq_len);   // first-digit histograms per row (IndexerArgs::hist_chunks)
// The two halves of topk_launch for rows scored a key span at a time: the chunk pass
// over chunks c0 .. c0+nl-1 of every row (scores: row t's key c0 * chunk_len at
// scores + t * stride), writing their lists into scratch; then the merge levels.
cudaError_t topk_chunks_launch(const GeomDev& g, const float* scores, int64_t stride, int k, int c0, int nl,
                               void* scratch, int* err, bool pdl, cudaStream_t st, int* hist = nullptr);
cudaError_t topk_merge_launch(const GeomDev& g, int k, int* idx, void* scratch, int* err, bool pdl, cudaStream_t st);

// ---- sparse MLA + combine (sparse_mla.cu)
struct MlaArgs {
  GeomDev g;
  int H;               // total heads
  int k;               // idx row length
  int C;               // chunks per query
  int64_t n_chunks;    // T * C
  const uint8_t* kv;   // paged latent cache
  const int* idx;      // [T, k]
  float scale_log2;    // sm_scale * log2(e)
  __nv_bfloat16* out;  // [T, H, 512]
  float* lse;          // [T, H] or null
  float* o_part;       // [T + G, H, 512]
  float* ml_part;      // [T + G, H, 2]  (running max in log2 units, sum)
  int* err;
};
// Number of two-CTA clusters of the persistent attention grid.
int mla_grid(int64_t n_chunks, int num_sms);
size_t mla_partial_bytes(int T, int H, int grid);
// map_q: [T*H, 576] bf16 query rows, 64 x min(H,16) box, 128-byte swizzle.
// Latent cache formats: bf16 rows of 576, or pages of 656-byte records (512 codes, e4m3
// or int8; four fp32 scales, one per 128 codes; 64 bf16 RoPE values) stored per page as
// code, scale and RoPE planes (common.cuh).
enum KvFormat : int { kKvBf16 = 0, kKvE4m3 = 1, kKvInt8 = 2 };
cudaError_t mla_launch(int kv_format, const CUtensorMap& map_q, MlaArgs A, int grid, bool pdl, cudaStream_t st);
bool encode_mla_q_map(CUtensorMap* map_q, const void* q, int T, int H);

// ---- cache append (cache_append.cu)
struct AppendArgs {
  GeomDev g;
  int kv_format;                // KvFormat of the latent cache
  const void* kv_new;           // [T, 576] bf16
  uint8_t* kv_cache;            // [P*64] rows
  bool k_fp8;                   // index keys: e4m3 + per-token scale (else bf16)
  const void* k_new;            // [T, 128] bf16, or null to leave the index cache alone
  uint8_t* k_cache;             // [P*64] rows of 128 e4m3 codes or 128 bf16
  float* k_scale;               // [P*64] (e4m3 keys)
  int* err;
};
cudaError_t cache_append_launch(const AppendArgs& A, cudaStream_t st);

// ---- query ranges (indexer.cu): for j < n, the range of queries [t_first + j*rows,
// + rows) of the geometry alone, with their positions unchanged, as cu_q [B+1] then
// seq_lens [B] at out + j*stride.
cudaError_t query_ranges_launch(const int* cu_q, const int* seq_lens, int B, int T, int t_first, int rows, int n,
                                int* out, int stride, cudaStream_t st);

// ---- staging copy (stage_copy.cu): `bytes` from src to dst by the SMs; both are
// device-visible addresses (device memory, or mapped page-locked host memory).
cudaError_t stage_copy_launch(void* dst, const void* src, size_t bytes, int num_sms, cudaStream_t st);

// ---- indexer preparation (indexer_prep.cu)
struct PrepArgs {
  GeomDev g;
  int Hi;                       // indexer heads
  int rope_dim;                 // rotated values at the front of each 128 (multiple of 8)
  int split;                    // blocks per token (each takes a run of whole 4-head groups)
  const void* q_in;             // [T, Hi, 128] bf16
  const void* k_in;             // [T, 128] bf16, or null (queries only)
  const float* rope_cos;        // [max_seq_len, rope_dim/2]
  const float* rope_sin;        // [max_seq_len, rope_dim/2]
  const float* ln_gamma;        // [128] or null (1)
  const float* ln_beta;         // [128] or null (0)
  float ln_eps;
  uint8_t* q_out;               // [T, Hi, 128] e4m3
  float* q_scale;               // [T, Hi]
  uint8_t* k_cache;             // [P*64, 128] e4m3
  float* k_scale;               // [P*64]
  int* err;
};
cudaError_t indexer_prep_launch(const PrepArgs& A, cudaStream_t st);

// ---- host helpers defined in api.cu
// Host-side argument checks shared by every entry point that takes these arguments.
dsa_status_t check_geom(const dsa_geom_t* g);
dsa_status_t check_attend(const dsa_geom_t* g, dsa_dtype_t dt, int H, const void* q, const void* kv, const int* idx,
                          int k, float sm_scale, const void* out);
// Device addresses of the attention's outputs: out [T, H, 512] bf16 and lse [T, H]
// fp32 (or null) may be device memory or page-locked host memory the device maps (the
// kernels then write the results straight to the host); anything else is refused.
dsa_status_t resolve_outputs(const dsa_geom_t* g, int H, void* out, float* lse, void** dout, float** dlse);
bool encode_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols,
                          uint64_t rows, uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows);
void set_last_error(const char* what, const char* detail);

}  // namespace dsa
