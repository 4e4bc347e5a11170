// dsa_sparse_mla_attend_static: the sparse-MLA entry point for callers that
// cannot hand the library device memory at call time -- a runtime whose device
// memory is planned and reserved up front, a plugin host that offers no
// workspace, or code at a point where an allocation would synchronize the
// device or disturb a memory pool. It takes no workspace: the split-softmax
// partials go to a file-scope static device buffer that the library owns.
//
// The buffer is kStaticScratchBytes per GPU, held by every GPU that loads the
// library until the process exits. Its address is looked up once per device
// (cudaGetSymbolAddress with that device current) on the first call there, so
// that first call should come before any stream capture. All calls share the
// buffer and it keeps the last call's contents; nothing in it needs to start at
// zero (every partial row a call reads was written earlier in the same call).
// Calls whose work overlaps on the GPU (other streams, other threads) race on it.
#include <cmath>
#include <cstdio>
#include <mutex>
#include "dsa.h"
#include "kernels.cuh"

namespace {

constexpr size_t kStaticScratchBytes = DSA_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};


// Device address of g_static_scratch on the current device (set up once per device).
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

using namespace dsa;

extern "C" dsa_status_t dsa_sparse_mla_attend_static(const dsa_geom_t* geom, dsa_dtype_t kv_dtype, int32_t H,
                                                     const void* q, const void* kv_cache, const int32_t* idx,
                                                     int32_t k, float sm_scale, void* out, float* lse,
                                                     int32_t* err_word, void* stream) {
  // the same argument rules as dsa_sparse_mla_attend
  const dsa_status_t s = check_attend(geom, kv_dtype, H, q, kv_cache, idx, k, sm_scale, out);
  if (s != DSA_OK) return s;
  // A bounded wait that gives up stops the kernel before it writes its partial rows,
  // and the merge then reads rows an earlier call left in the shared buffer: the
  // error word is what reports that, so it is required here.
  if (!err_word || (reinterpret_cast<uintptr_t>(err_word) & 3u)) return DSA_ERR_INVALID_ARG;
  if (geom->T == 0) return DSA_OK;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DSA_ERR_CUDA;
  MlaArgs A;
  A.H = H; A.k = k; A.C = (k + 127) / 128; A.n_chunks = (int64_t)geom->T * A.C;
  const int grid = mla_grid(A.n_chunks, sms);
  const size_t need = mla_partial_bytes(geom->T, H, grid);
  if (need > kStaticScratchBytes) {
    char buf[160];
    snprintf(buf, sizeof(buf), "static scratch holds %zu bytes; T=%d, H=%d need %zu", kStaticScratchBytes,
             geom->T, H, need);
    set_last_error("dsa_sparse_mla_attend_static", buf);
    return DSA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const cudaError_t se = scratch_address(&scratch);
  if (se != cudaSuccess) {
    set_last_error("cudaGetSymbolAddress", cudaGetErrorString(se));
    return DSA_ERR_CUDA;
  }
  void* dout = nullptr;
  float* dlse = nullptr;
  const dsa_status_t rs = resolve_outputs(geom, H, out, lse, &dout, &dlse);
  if (rs != DSA_OK) return rs;
  CUtensorMap mq;
  if (!encode_mla_q_map(&mq, q, geom->T, H)) return DSA_ERR_CUDA;
  A.g.B = geom->B; A.g.T = geom->T; A.g.max_seq_len = geom->max_seq_len; A.g.num_pages = geom->num_pages;
  A.g.bt_stride = geom->bt_stride; A.g.seq_lens = geom->seq_lens; A.g.cu_q = geom->cu_q;
  A.g.block_table = geom->block_table;
  A.kv = reinterpret_cast<const uint8_t*>(kv_cache); A.idx = idx; A.scale_log2 = sm_scale * 1.4426950408889634f;
  A.out = reinterpret_cast<__nv_bfloat16*>(dout); A.lse = dlse;
  A.o_part = reinterpret_cast<float*>(scratch);
  A.ml_part = A.o_part + (size_t)(geom->T + grid) * H * 512;
  A.err = reinterpret_cast<int*>(err_word);
  const int kv_format = kv_dtype == DSA_E4M3 ? kKvE4m3 : kv_dtype == DSA_I8 ? kKvInt8 : kKvBf16;
  const cudaError_t le = mla_launch(kv_format, mq, A, grid, false, reinterpret_cast<cudaStream_t>(stream));
  if (le != cudaSuccess) {
    set_last_error("kernel launch", cudaGetErrorString(le));
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}
