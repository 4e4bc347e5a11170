// Host side of the C ABI declared in include/dsa.h: argument validation,
// workspace layout, TMA descriptor encoding and kernel launches.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include "dsa.h"
#include "kernels.cuh"


using namespace dsa;

namespace dsa {

thread_local char g_last_error[256] = "";

void set_last_error(const char* what, const char* detail) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, detail);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D row-major tensor [rows, cols] with a 128-byte-swizzled box of box_cols x box_rows.
bool encode_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
               uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) { set_last_error("cudaGetDriverEntryPointByVersion", "cuTensorMapEncodeTiled unavailable"); return false; }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    snprintf(buf, sizeof(buf), "CUresult %d (dims %llu x %llu, box %u x %u)", (int)r, (unsigned long long)cols,
             (unsigned long long)rows, box_cols, box_rows);
    set_last_error("cuTensorMapEncodeTiled", buf);
    return false;
  }
  return true;
}

bool encode_mla_q_map(CUtensorMap* map_q, const void* q, int T, int H) {
  const uint32_t box_rows = H < 16 ? (uint32_t)H : 16u;
  return encode_tensor_map_2d(map_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, 576, (uint64_t)T * H, 1152, 64, box_rows);
}

}  // namespace dsa

namespace {

constexpr size_t kHeaderBytes = 256;
constexpr int kMaxTopk = 16384;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int kv_format_of(dsa_dtype_t dt) { return dt == DSA_E4M3 ? kKvE4m3 : dt == DSA_I8 ? kKvInt8 : kKvBf16; }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

}  // namespace

namespace dsa {

dsa_status_t check_geom(const dsa_geom_t* g) {
  if (!g) return DSA_ERR_INVALID_ARG;
  if (g->B < 0 || g->T < 0 || g->max_seq_len < 1 || g->num_pages < 1) return DSA_ERR_INVALID_ARG;
  if (g->page_size != 64) return DSA_ERR_UNSUPPORTED;
  if (g->T > 0 && g->B < 1) return DSA_ERR_INVALID_ARG;
  if (g->bt_stride < (g->max_seq_len + 63) / 64) return DSA_ERR_INVALID_ARG;
  if ((int64_t)g->num_pages * 64 > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if (g->B > 0 && (!g->seq_lens || !g->cu_q || !g->block_table)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

dsa_status_t check_attend(const dsa_geom_t* g, dsa_dtype_t dt, int H, const void* q, const void* kv, const int* idx,
                          int k, float sm_scale, const void* out) {
  dsa_status_t s = check_geom(g);
  if (s != DSA_OK) return s;
  if (dt != DSA_BF16 && dt != DSA_E4M3 && dt != DSA_I8) return DSA_ERR_INVALID_ARG;
  if (H < 1 || H > 128 || (H > 16 && H % 16 != 0)) return DSA_ERR_INVALID_ARG;
  if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return DSA_ERR_INVALID_ARG;
  if (g->T == 0) return DSA_OK;
  if (!q || !kv || !idx || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// Device-visible address of the range [p, p + bytes): device or managed memory, or
// page-locked host memory the device maps; both ends must resolve to one contiguous
// mapping. Anything else (pageable host memory, unknown pointers) is refused.
bool device_range(const void* p, size_t bytes, const void** out) {
  cudaPointerAttributes a0, a1;
  const void* last = reinterpret_cast<const uint8_t*>(p) + (bytes - 1);
  if (cudaPointerGetAttributes(&a0, p) != cudaSuccess || cudaPointerGetAttributes(&a1, last) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  auto visible = [](const cudaPointerAttributes& a) {
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
           (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr);
  };
  if (!visible(a0) || !visible(a1) || a0.type != a1.type || a0.device != a1.device) return false;
  const uint8_t* d0 = reinterpret_cast<const uint8_t*>(a0.devicePointer ? a0.devicePointer : p);
  const uint8_t* d1 = reinterpret_cast<const uint8_t*>(a1.devicePointer ? a1.devicePointer : last);
  if (d1 != d0 + (bytes - 1)) return false;
  *out = d0;
  return true;
}


dsa_status_t resolve_outputs(const dsa_geom_t* g, int H, void* out, float* lse, void** dout, float** dlse) {
  const void* o = nullptr;
  const void* l = nullptr;
  if (!device_range(out, (size_t)g->T * H * 512 * 2, &o) || (lse && !device_range(lse, (size_t)g->T * H * 4, &l))) {
    set_last_error("sparse MLA outputs", "out and lse must be device memory or page-locked host memory the device maps");
    return DSA_ERR_INVALID_ARG;
  }
  *dout = const_cast<void*>(o);
  *dlse = reinterpret_cast<float*>(const_cast<void*>(l));
  return DSA_OK;
}

}  // namespace dsa

namespace {

GeomDev to_dev(const dsa_geom_t* g) {
  GeomDev d;
  d.B = g->B; d.T = g->T; d.max_seq_len = g->max_seq_len; d.num_pages = g->num_pages; d.bt_stride = g->bt_stride;
  d.seq_lens = g->seq_lens; d.cu_q = g->cu_q; d.block_table = g->block_table;
  return d;
}

dsa_status_t from_cuda(cudaError_t e, const char* what = "kernel launch") {
  if (e == cudaSuccess) return DSA_OK;
  set_last_error(what, cudaGetErrorString(e));
  return DSA_ERR_CUDA;
}

// ---------------------------------------------------------------- indexer
dsa_status_t check_indexer(const dsa_geom_t* g, dsa_dtype_t dt, int Hi, const void* q_idx, const float* q_scale,
                           const float* w, const void* kc, const float* ks, const float* scores, int64_t stride) {
  dsa_status_t s = check_geom(g);
  if (s != DSA_OK) return s;
  if (dt != DSA_BF16 && dt != DSA_E4M3) return DSA_ERR_INVALID_ARG;
  if (Hi < 1 || Hi > 64) return DSA_ERR_INVALID_ARG;
  if (stride < g->max_seq_len) return DSA_ERR_INVALID_ARG;
  if (g->T == 0) return DSA_OK;
  if (!q_idx || !w || !kc || !scores) return DSA_ERR_INVALID_ARG;
  if (dt == DSA_E4M3 && (!q_scale || !ks)) return DSA_ERR_INVALID_ARG;
  if (dt == DSA_BF16 && (q_scale || ks)) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(kc) || !aligned16(w)) return DSA_ERR_INVALID_ARG;
  if (dt == DSA_E4M3 && (!aligned16(q_scale) || !aligned16(ks))) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// Scores of keys [key_begin, key_end) (multiples of 128; key_end past every length for
// all keys) into column s - key_begin of `scores`. The kernel holds the metadata of up
// to indexer_max_requests() requests; more are scored in groups of that many, one
// launch each (query rows stay absolute: each group's cu_q entries index them).
dsa_status_t run_indexer(const dsa_geom_t* g, dsa_dtype_t dt, int Hi, const void* q_idx, const float* q_scale,
                         const float* w, const void* kc, const float* ks, float* scores, int64_t stride, int* err,
                         cudaStream_t st, int key_begin = 0, int key_end = INT32_MAX, bool pdl = false,
                         int* hist = nullptr) {
  const bool fp8 = dt == DSA_E4M3;
  CUtensorMap mk, mq;
  const CUtensorMapDataType tdt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t box_cols = fp8 ? 128 : 64;
  const uint64_t row_bytes = fp8 ? 128 : 256;
  if (!encode_tensor_map_2d(&mk, tdt, kc, 128, (uint64_t)g->num_pages * 64, row_bytes, box_cols, 64)) return DSA_ERR_CUDA;
  const bool multi = g->T > g->B;   // some request has more than one query token
  const int q_box = indexer_q_box_rows(Hi, multi);
  if (!encode_tensor_map_2d(&mq, tdt, q_idx, 128, (uint64_t)g->T * Hi, row_bytes, box_cols, (uint32_t)q_box))
    return DSA_ERR_CUDA;
  IndexerArgs A;
  A.q_group_box = q_box != Hi;
  A.Hi = Hi; A.q_scale = q_scale; A.w = w; A.k_scale = ks; A.scores = scores; A.stride = stride;
  A.key_begin = key_begin; A.key_end = key_end;
  A.hist = hist; A.hist_chunks = topk_row_chunks(g->max_seq_len);
  A.err = err;
  const int group = indexer_max_requests();
  for (int b0 = 0; b0 < g->B; b0 += group) {
    dsa_geom_t sub = *g;
    sub.B = g->B - b0 < group ? g->B - b0 : group;
    sub.seq_lens = g->seq_lens + b0;
    sub.cu_q = g->cu_q + b0;
    sub.block_table = g->block_table + (int64_t)b0 * g->bt_stride;
    A.g = to_dev(&sub);
    const dsa_status_t s = from_cuda(indexer_launch(fp8, Hi, multi, mk, mq, A, num_sms(), pdl || b0 > 0, st));
    if (s != DSA_OK) return s;
  }
  return DSA_OK;
}

// ---------------------------------------------------------------- top-k
dsa_status_t check_topk(const dsa_geom_t* g, const float* scores, int64_t stride, int k, const int* idx) {
  dsa_status_t s = check_geom(g);
  if (s != DSA_OK) return s;
  if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
  if (stride < g->max_seq_len) return DSA_ERR_INVALID_ARG;
  if (topk_merge_levels(g->max_seq_len, k) < 0) {
    set_last_error("dsa_topk", "rows longer than 16384 positions need index_topk <= 8192");
    return DSA_ERR_UNSUPPORTED;
  }
  if (g->T == 0) return DSA_OK;
  if (!scores || !idx) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// ---------------------------------------------------------------- attention
size_t attend_scratch_bytes(const dsa_geom_t* g, int H, int k) {
  const int64_t C = (k + 127) / 128;
  const int grid = mla_grid((int64_t)g->T * C, num_sms());
  return mla_partial_bytes(g->T, H, grid);
}

dsa_status_t run_attend(const dsa_geom_t* g, dsa_dtype_t dt, int H, const void* q, const void* kv, const int* idx,
                        int k, float sm_scale, void* out, float* lse, void* scratch, int* err, bool pdl,
                        cudaStream_t st) {
  void* dout = nullptr;
  float* dlse = nullptr;
  const dsa_status_t rs = resolve_outputs(g, H, out, lse, &dout, &dlse);
  if (rs != DSA_OK) return rs;
  CUtensorMap mq;
  if (!encode_mla_q_map(&mq, q, g->T, H)) return DSA_ERR_CUDA;
  MlaArgs A;
  A.g = to_dev(g); A.H = H; A.k = k; A.C = (k + 127) / 128; A.n_chunks = (int64_t)g->T * A.C;
  A.kv = reinterpret_cast<const uint8_t*>(kv); A.idx = idx; A.scale_log2 = sm_scale * 1.4426950408889634f;
  A.out = reinterpret_cast<__nv_bfloat16*>(dout); A.lse = dlse;
  const int grid = mla_grid(A.n_chunks, num_sms());
  const size_t rows = (size_t)(g->T + grid) * H;
  A.o_part = reinterpret_cast<float*>(scratch);
  A.ml_part = A.o_part + rows * 512;
  A.err = err;
  return from_cuda(mla_launch(kv_format_of(dt), mq, A, grid, pdl, st));
}

int64_t step_score_stride(const dsa_geom_t* g) { return (int64_t)align_up((size_t)g->max_seq_len, 64); }

}  // namespace

extern "C" {

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported argument combination";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_TIMEOUT: return "device wait timed out";
    case DSA_ERR_WORKSPACE: return "workspace too small or misaligned";
    case DSA_ERR_BAD_INDEX: return "device data out of range (page id, index or sequence geometry)";
  }
  return "unknown status";
}

int32_t dsa_abi_version(void) { return DSA_ABI_VERSION; }

const char* dsa_last_error(void) { return g_last_error; }

size_t dsa_indexer_scores_workspace_size(const dsa_geom_t*) { return kHeaderBytes; }

dsa_status_t dsa_indexer_scores(const dsa_geom_t* geom, dsa_dtype_t qk_dtype, int32_t Hi, const void* q_idx,
                                const float* q_scale, const float* w, const void* idx_k_cache,
                                const float* idx_k_scale, float* scores, int64_t score_stride, void* ws,
                                size_t ws_bytes, void* stream) {
  dsa_status_t s = check_indexer(geom, qk_dtype, Hi, q_idx, q_scale, w, idx_k_cache, idx_k_scale, scores, score_stride);
  if (s != DSA_OK) return s;
  if (!ws || ws_bytes < kHeaderBytes || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DSA_ERR_WORKSPACE;
  if (geom->T == 0 || geom->B == 0) return DSA_OK;
  return run_indexer(geom, qk_dtype, Hi, q_idx, q_scale, w, idx_k_cache, idx_k_scale, scores, score_stride,
                     reinterpret_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream));
}

size_t dsa_topk_workspace_size(const dsa_geom_t* geom, int32_t k) {
  if (!geom || k < 1) return kHeaderBytes;
  return kHeaderBytes + align_up(topk_workspace_bytes(geom->T, geom->max_seq_len, k), 256);
}

dsa_status_t dsa_topk(const dsa_geom_t* geom, const float* scores, int64_t score_stride, int32_t k, int32_t* idx,
                      void* ws, size_t ws_bytes, void* stream) {
  dsa_status_t s = check_topk(geom, scores, score_stride, k, idx);
  if (s != DSA_OK) return s;
  if (!ws || ws_bytes < dsa_topk_workspace_size(geom, k) || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return DSA_ERR_WORKSPACE;
  if (geom->T == 0) return DSA_OK;
  return from_cuda(topk_launch(to_dev(geom), scores, score_stride, k, idx,
                               reinterpret_cast<uint8_t*>(ws) + kHeaderBytes, reinterpret_cast<int*>(ws), false,
                               reinterpret_cast<cudaStream_t>(stream)));
}

size_t dsa_sparse_mla_attend_workspace_size(const dsa_geom_t* geom, int32_t H, int32_t k) {
  if (!geom || H < 1 || k < 1) return kHeaderBytes;
  return kHeaderBytes + align_up(attend_scratch_bytes(geom, H, k), 256);
}

dsa_status_t dsa_sparse_mla_attend(const dsa_geom_t* geom, dsa_dtype_t kv_dtype, int32_t H, const void* q,
                                   const void* kv_cache, const int32_t* idx, int32_t k, float sm_scale, void* out,
                                   float* lse, void* ws, size_t ws_bytes, void* stream) {
  dsa_status_t s = check_attend(geom, kv_dtype, H, q, kv_cache, idx, k, sm_scale, out);
  if (s != DSA_OK) return s;
  if (!ws || ws_bytes < dsa_sparse_mla_attend_workspace_size(geom, H, k) || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return DSA_ERR_WORKSPACE;
  if (geom->T == 0) return DSA_OK;
  return run_attend(geom, kv_dtype, H, q, kv_cache, idx, k, sm_scale, out, lse,
                    reinterpret_cast<uint8_t*>(ws) + kHeaderBytes, reinterpret_cast<int*>(ws), false,
                    reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// How the step holds its scores: `rows` queries at a time (rows >= T: all at once),
// each over keys in spans of `span` positions (0: whole rows). A span is a multiple
// of the top-k chunk length, so every chunk of a row is scored within one span.
struct ScorePlan {
  int64_t rows;
  int64_t span;
};

ScorePlan whole_rows(const dsa_step_args_t* a) { return ScorePlan{a->geom.T, 0}; }

// Width of the score buffer's rows.
int64_t plan_width(const dsa_geom_t* g, const ScorePlan& p) { return p.span > 0 ? p.span : step_score_stride(g); }

// Query ranges of the bounded step: the geometry of up to kRangeRing ranges is written
// by one launch before the first of them, each range's in a slot of range_stride ints
// (a few KB, small beside even a one-row score budget).
constexpr int kRangeRing = 8;
int range_stride(const dsa_geom_t* g) { return (2 * g->B + 1 + 3) / 4 * 4; }
size_t range_ring_bytes(const dsa_geom_t* g, int64_t rows) {
  const int64_t n = (g->T + rows - 1) / rows;
  return align_up((size_t)(n < kRangeRing ? n : kRangeRing) * range_stride(g) * sizeof(int32_t), 256);
}

// Whole rows at once, when asked for: the indexer also counts the top-k's first-digit
// histograms.
bool plan_hist(const dsa_geom_t* g, const ScorePlan& p, bool hist) { return hist && p.rows >= g->T && p.span == 0; }

// Workspace of the step under a score plan. Layout: header | query-range geometry
// (ranges only) | scores [rows, width] | idx [T, k] (unless idx_out) | attention /
// top-k scratch | first-digit histograms (whole rows only). The histograms come last:
// the top-k leaves them zero for the next step, and a shared layer's step on the same
// workspace (header | scratch) stays clear of them.
size_t step_workspace_bytes(const dsa_step_args_t* a, const ScorePlan& p, bool hist = false) {
  const dsa_geom_t* g = &a->geom;
  size_t bytes = kHeaderBytes;
  const int64_t r = p.rows < g->T ? p.rows : g->T;
  if (!a->reuse_idx) {
    if (r < g->T) bytes += range_ring_bytes(g, r);
    bytes += align_up((size_t)r * plan_width(g, p) * sizeof(float), 256);
    if (!a->idx_out) bytes += align_up((size_t)g->T * (a->topk > 0 ? a->topk : 1) * sizeof(int32_t), 256);
  }
  size_t scratch = attend_scratch_bytes(g, a->H > 0 ? a->H : 1, a->topk > 0 ? a->topk : 1);
  if (!a->reuse_idx && a->topk > 0) {
    const size_t tk = topk_workspace_bytes((int)r, g->max_seq_len, a->topk);
    if (tk > scratch) scratch = tk;
  }
  bytes += align_up(scratch, 256);
  if (!a->reuse_idx && plan_hist(g, p, hist)) bytes += align_up(topk_hist_bytes(g->T, g->max_seq_len), 256);
  return bytes;
}

// Scores and selects one range of queries (geometry `sub`, whose rows are the step's
// rows t0.. onward) into idx_out: the whole rows at once, or span by span, each
// span's chunks reduced to candidate lists before the next span is scored.
// pdl_first: the range's first indexer launch may start before the kernel just before
// it ends (that kernel is our own and the range's geometry is already written).
// hist: first-digit histograms for whole rows (p.span == 0), or null.
dsa_status_t select_range(const dsa_step_args_t* a, const dsa_geom_t* sub, int64_t t0, const ScorePlan& p,
                          float* scores, int32_t* idx_out, void* scratch, int* err, bool pdl_first, cudaStream_t st,
                          int* hist = nullptr) {
  const dsa_geom_t* g = &a->geom;
  const size_t qrow = (size_t)a->Hi * 128 * (a->qk_dtype == DSA_E4M3 ? 1 : 2);
  const uint8_t* q_idx = reinterpret_cast<const uint8_t*>(a->q_idx) + (size_t)t0 * qrow;
  const float* q_scale = a->q_scale ? a->q_scale + (size_t)t0 * a->Hi : nullptr;
  const float* w = a->w + (size_t)t0 * a->Hi;
  dsa_status_t s;
  if (p.span == 0) {
    const int64_t stride = step_score_stride(g);
    s = run_indexer(sub, a->qk_dtype, a->Hi, q_idx, q_scale, w, a->idx_k_cache, a->idx_k_scale, scores, stride, err, st,
                    0, INT32_MAX, pdl_first, hist);
    if (s != DSA_OK) return s;
    // The top-k kernels follow this call's own kernels, so they may launch early
    // (programmatic dependent launch) and wait for their inputs inside.
    return from_cuda(topk_launch(to_dev(sub), scores, stride, a->topk, idx_out, scratch, err, true, st, hist));
  }
  const int chunk = topk_chunk_len();
  const int nch = (g->max_seq_len + chunk - 1) / chunk;
  const int per_span = (int)(p.span / chunk);
  for (int c0 = 0; c0 < nch; c0 += per_span) {
    const int nl = nch - c0 < per_span ? nch - c0 : per_span;
    const int64_t k0 = (int64_t)c0 * chunk;
    // a later span's scores overwrite the buffer only after its grid-dependency wait,
    // which the previous span's chunk pass ends
    s = run_indexer(sub, a->qk_dtype, a->Hi, q_idx, q_scale, w, a->idx_k_cache, a->idx_k_scale, scores, p.span, err,
                    st, (int)k0, (int)(k0 + p.span < INT32_MAX ? k0 + p.span : INT32_MAX), pdl_first || c0 > 0);
    if (s != DSA_OK) return s;
    s = from_cuda(topk_chunks_launch(to_dev(sub), scores, p.span, a->topk, c0, nl, scratch, err, true, st));
    if (s != DSA_OK) return s;
  }
  return from_cuda(topk_merge_launch(to_dev(sub), a->topk, idx_out, scratch, err, true, st));
}

// The step with the queries' scores held as the plan says (the selection of each
// query does not depend on the others', and a span's chunk lists are those the whole
// row gives, so the result is the same for every plan).
dsa_status_t run_step(const dsa_step_args_t* a, const ScorePlan& p, void* ws, size_t ws_bytes, void* stream,
                      cudaEvent_t q_ready = nullptr, bool hist = false) {
  const dsa_geom_t* g = &a->geom;
  dsa_status_t s;
  if (!a->reuse_idx) {
    s = check_indexer(g, a->qk_dtype, a->Hi, a->q_idx, a->q_scale, a->w, a->idx_k_cache, a->idx_k_scale,
                      reinterpret_cast<const float*>(ws), step_score_stride(g));
    if (s != DSA_OK) return s;
    s = check_topk(g, reinterpret_cast<const float*>(ws), step_score_stride(g), a->topk, reinterpret_cast<const int*>(ws));
    if (s != DSA_OK) return s;
  }
  s = check_attend(g, a->kv_dtype, a->H, a->q, a->kv_cache, a->reuse_idx ? a->reuse_idx : reinterpret_cast<const int*>(ws),
                   a->topk, a->sm_scale, a->out);
  if (s != DSA_OK) return s;
  if (!ws || ws_bytes < step_workspace_bytes(a, p, hist) || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return DSA_ERR_WORKSPACE;
  if (g->T == 0) return DSA_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ptr = reinterpret_cast<uint8_t*>(ws);
  int* err = reinterpret_cast<int*>(ws);
  ptr += kHeaderBytes;
  const int32_t* idx = a->reuse_idx;
  if (!idx) {
    const bool ranges = p.rows < g->T;
    int32_t* range_geom = nullptr;
    if (ranges) {
      range_geom = reinterpret_cast<int32_t*>(ptr);
      ptr += range_ring_bytes(g, p.rows);
    }
    const int64_t r = ranges ? p.rows : g->T;
    float* scores = reinterpret_cast<float*>(ptr);
    ptr += align_up((size_t)r * plan_width(g, p) * sizeof(float), 256);
    int32_t* idx_buf = a->idx_out;
    if (!idx_buf) {
      idx_buf = reinterpret_cast<int32_t*>(ptr);
      ptr += align_up((size_t)g->T * a->topk * sizeof(int32_t), 256);
    }
    if (!ranges) {
      int* hist_buf = nullptr;
      if (plan_hist(g, p, hist) && indexer_counts_hist(a->qk_dtype == DSA_E4M3, a->Hi, g->T > g->B))
        hist_buf = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ws) + step_workspace_bytes(a, p, true) -
                                          align_up(topk_hist_bytes(g->T, g->max_seq_len), 256));
      s = select_range(a, g, 0, p, scores, idx_buf, ptr, err, false, st, hist_buf);
      if (s != DSA_OK) return s;
    } else {
      // Bounded scoring: queries [t0, t0 + rows) at a time, each range described by
      // its own geometry (same requests, block table and positions), scored into the
      // same rows of `scores` and reduced to its selection before the next range. The
      // geometries of up to kRangeRing ranges are written by one launch ahead of them,
      // so each later range's indexer may start (programmatic dependent launch) while
      // the previous range's top-k finishes; its scores wait for it.
      const int stride = range_stride(g);
      const int64_t n_ranges = (g->T + p.rows - 1) / p.rows;
      for (int64_t r = 0; r < n_ranges; ++r) {
        const int64_t t0 = r * p.rows;
        const int t1 = (int)(t0 + p.rows < g->T ? t0 + p.rows : g->T);
        const int slot = (int)(r % kRangeRing);
        if (slot == 0) {
          const int n = (int)(n_ranges - r < kRangeRing ? n_ranges - r : kRangeRing);
          s = from_cuda(query_ranges_launch(g->cu_q, g->seq_lens, g->B, g->T, (int)t0, (int)p.rows, n, range_geom,
                                            stride, st));
          if (s != DSA_OK) return s;
        }
        dsa_geom_t sub = *g;
        sub.T = t1 - (int)t0;
        sub.cu_q = range_geom + (size_t)slot * stride;
        sub.seq_lens = sub.cu_q + g->B + 1;
        s = select_range(a, &sub, t0, p, scores, idx_buf + (size_t)t0 * a->topk, ptr, err, slot != 0, st);
        if (s != DSA_OK) return s;
      }
    }
    idx = idx_buf;
  }
  // The MLA query may still be arriving (its copy recorded q_ready): the attention
  // waits for it, the indexer and top-k above did not. Its launch then waits on the
  // event as a whole instead of overlapping the top-k's tail.
  if (q_ready) {
    s = from_cuda(cudaStreamWaitEvent(st, q_ready, 0));
    if (s != DSA_OK) return s;
  }
  return run_attend(g, a->kv_dtype, a->H, a->q, a->kv_cache, idx, a->topk, a->sm_scale, a->out, a->lse, ptr, err,
                    a->reuse_idx == nullptr && q_ready == nullptr, st);
}

}  // namespace

extern "C" {

size_t dsa_decode_step_workspace_size(const dsa_step_args_t* a) {
  if (!a) return kHeaderBytes;
  return step_workspace_bytes(a, whole_rows(a));
}

dsa_status_t dsa_decode_step(const dsa_step_args_t* a, void* ws, size_t ws_bytes, void* stream) {
  if (!a) return DSA_ERR_INVALID_ARG;
  return run_step(a, whole_rows(a), ws, ws_bytes, stream);
}

dsa_status_t dsa_decode_step_wait_q(const dsa_step_args_t* a, void* q_ready, void* ws, size_t ws_bytes, void* stream) {
  if (!a) return DSA_ERR_INVALID_ARG;
  return run_step(a, whole_rows(a), ws, ws_bytes, stream, reinterpret_cast<cudaEvent_t>(q_ready));
}

size_t dsa_decode_step_hist_workspace_size(const dsa_step_args_t* a) {
  if (!a) return kHeaderBytes;
  return step_workspace_bytes(a, whole_rows(a), true);
}

dsa_status_t dsa_decode_step_hist(const dsa_step_args_t* a, void* ws, size_t ws_bytes, void* stream) {
  if (!a) return DSA_ERR_INVALID_ARG;
  return run_step(a, whole_rows(a), ws, ws_bytes, stream, nullptr, true);
}

// The score plan a budget allows: as many whole rows as fit; below one row, one query
// at a time over spans of whole top-k chunks. rows == 0: not even one chunk fits.
static ScorePlan bounded_plan(const dsa_step_args_t* a, size_t score_budget_bytes) {
  const size_t row = (size_t)step_score_stride(&a->geom) * sizeof(float);
  if (score_budget_bytes >= row) return ScorePlan{(int64_t)(score_budget_bytes / row), 0};
  const size_t chunk = (size_t)topk_chunk_len();
  const int64_t span = (int64_t)(score_budget_bytes / (chunk * sizeof(float)) * chunk);
  return span > 0 ? ScorePlan{1, span} : ScorePlan{0, 0};
}

size_t dsa_decode_step_bounded_workspace_size(const dsa_step_args_t* a, size_t score_budget_bytes) {
  if (!a) return kHeaderBytes;
  const ScorePlan p = bounded_plan(a, score_budget_bytes);
  return step_workspace_bytes(a, p.rows < 1 ? ScorePlan{1, 0} : p);
}

dsa_status_t dsa_decode_step_bounded(const dsa_step_args_t* a, size_t score_budget_bytes, void* ws, size_t ws_bytes,
                                     void* stream) {
  if (!a) return DSA_ERR_INVALID_ARG;
  const ScorePlan p = bounded_plan(a, score_budget_bytes);
  if (p.rows < 1 && !a->reuse_idx) {
    char buf[192];
    snprintf(buf, sizeof(buf),
             "score budget %zu bytes holds neither one query's score row (%zu bytes) nor one top-k chunk (%zu bytes)",
             score_budget_bytes, (size_t)step_score_stride(&a->geom) * sizeof(float),
             (size_t)topk_chunk_len() * sizeof(float));
    set_last_error("dsa_decode_step_bounded", buf);
    return DSA_ERR_INVALID_ARG;
  }
  return run_step(a, p.rows < 1 ? ScorePlan{1, 0} : p, ws, ws_bytes, stream);
}

size_t dsa_cache_append_workspace_size(const dsa_geom_t*) { return kHeaderBytes; }

dsa_status_t dsa_cache_append(const dsa_geom_t* geom, dsa_dtype_t kv_dtype, const void* kv_new, void* kv_cache,
                              dsa_dtype_t qk_dtype, const void* k_new, void* idx_k_cache, float* idx_k_scale,
                              void* ws, size_t ws_bytes, void* stream) {
  dsa_status_t s = check_geom(geom);
  if (s != DSA_OK) return s;
  if (kv_dtype != DSA_BF16 && kv_dtype != DSA_E4M3 && kv_dtype != DSA_I8) return DSA_ERR_INVALID_ARG;
  if (k_new) {
    if (qk_dtype != DSA_BF16 && qk_dtype != DSA_E4M3) return DSA_ERR_INVALID_ARG;
    if (!idx_k_cache || !aligned16(k_new) || !aligned16(idx_k_cache)) return DSA_ERR_INVALID_ARG;
    if (qk_dtype == DSA_E4M3 && !idx_k_scale) return DSA_ERR_INVALID_ARG;
    if (qk_dtype == DSA_BF16 && idx_k_scale) return DSA_ERR_INVALID_ARG;
  }
  if (!ws || ws_bytes < kHeaderBytes || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DSA_ERR_WORKSPACE;
  if (geom->T == 0) return DSA_OK;
  if (!kv_new || !kv_cache || !aligned16(kv_new) || !aligned16(kv_cache)) return DSA_ERR_INVALID_ARG;
  AppendArgs A;
  A.g = to_dev(geom);
  A.kv_format = kv_format_of(kv_dtype);
  A.kv_new = kv_new;
  A.kv_cache = reinterpret_cast<uint8_t*>(kv_cache);
  A.k_fp8 = qk_dtype == DSA_E4M3;
  A.k_new = k_new;
  A.k_cache = reinterpret_cast<uint8_t*>(idx_k_cache);
  A.k_scale = idx_k_scale;
  A.err = reinterpret_cast<int*>(ws);
  return from_cuda(cache_append_launch(A, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

}  // namespace

extern "C" {

dsa_status_t dsa_stage_copy(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return DSA_OK;
  if (!dst || !src || !aligned16(dst) || !aligned16(src)) return DSA_ERR_INVALID_ARG;
  const void *d = nullptr, *s = nullptr;
  if (!device_range(dst, bytes, &d) || !device_range(src, bytes, &s)) {
    set_last_error("dsa_stage_copy", "both ranges must be device memory or page-locked host memory the device maps");
    return DSA_ERR_INVALID_ARG;
  }
  if (!aligned16(d) || !aligned16(s)) return DSA_ERR_INVALID_ARG;
  return from_cuda(stage_copy_launch(const_cast<void*>(d), s, bytes, num_sms(), reinterpret_cast<cudaStream_t>(stream)));
}

size_t dsa_indexer_prepare_workspace_size(const dsa_geom_t*) { return kHeaderBytes; }

dsa_status_t dsa_indexer_prepare(const dsa_geom_t* geom, int32_t Hi, int32_t rope_dim, const void* q_in,
                                 const void* k_in, const float* rope_cos, const float* rope_sin,
                                 const float* ln_gamma, const float* ln_beta, float ln_eps, void* q_out,
                                 float* q_scale, void* idx_k_cache, float* idx_k_scale, void* ws, size_t ws_bytes,
                                 void* stream) {
  dsa_status_t s = check_geom(geom);
  if (s != DSA_OK) return s;
  if (Hi < 1 || Hi > 128) return DSA_ERR_INVALID_ARG;
  if (rope_dim < 8 || rope_dim > 128 || rope_dim % 8 != 0) return DSA_ERR_INVALID_ARG;
  if (!(ln_eps >= 0.f) || !std::isfinite(ln_eps)) return DSA_ERR_INVALID_ARG;
  if (k_in && (!idx_k_cache || !idx_k_scale || !aligned16(k_in) || !aligned16(idx_k_cache))) return DSA_ERR_INVALID_ARG;
  if ((ln_gamma && !aligned16(ln_gamma)) || (ln_beta && !aligned16(ln_beta))) return DSA_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kHeaderBytes || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DSA_ERR_WORKSPACE;
  if (geom->T == 0) return DSA_OK;
  if (!q_in || !q_out || !q_scale || !rope_cos || !rope_sin) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_in) || !aligned16(q_out) || !aligned16(rope_cos) || !aligned16(rope_sin)) return DSA_ERR_INVALID_ARG;
  PrepArgs A;
  A.g = to_dev(geom);
  A.Hi = Hi;
  A.rope_dim = rope_dim;
  // fewer tokens than two per SM: a token's heads are spread over up to 8 blocks
  {
    const int groups = (Hi + 3) / 4;
    int split = (2 * num_sms() + geom->T - 1) / geom->T;
    split = split < 1 ? 1 : (split > 8 ? 8 : split);
    A.split = split < groups ? split : groups;
  }
  A.q_in = q_in;
  A.k_in = k_in;
  A.rope_cos = rope_cos;
  A.rope_sin = rope_sin;
  A.ln_gamma = ln_gamma;
  A.ln_beta = ln_beta;
  A.ln_eps = ln_eps;
  A.q_out = reinterpret_cast<uint8_t*>(q_out);
  A.q_scale = q_scale;
  A.k_cache = reinterpret_cast<uint8_t*>(idx_k_cache);
  A.k_scale = idx_k_scale;
  A.err = reinterpret_cast<int*>(ws);
  return from_cuda(indexer_prep_launch(A, reinterpret_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_get_error(void* ws, void* stream) {
  if (!ws) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return from_cuda(e, "cudaStreamSynchronize");
  int code = 0;
  e = cudaMemcpy(&code, ws, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return from_cuda(e, "cudaMemcpy");
  if (code != 0) {
    e = cudaMemset(ws, 0, sizeof(int));
    if (e != cudaSuccess) return from_cuda(e, "cudaMemset");
  }
  return static_cast<dsa_status_t>(code);
}

dsa_status_t dsa_clear_error(void* ws, void* stream) {
  if (!ws) return DSA_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(ws, 0, kHeaderBytes, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
