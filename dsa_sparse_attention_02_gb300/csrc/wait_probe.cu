// dsa_wait_probe: the failure path of the bounded pipeline waits, run on purpose.
//
// Every wait of the library's kernels (an mbarrier phase that a copy, an MMA or
// another warp completes) gives up after a time limit, records DSA_ERR_TIMEOUT in
// the workspace's error word and returns, so that a stalled pipeline ends as a
// status the host reads instead of a hung context. This entry point exercises that
// path: one thread initializes an mbarrier that expects one arrival, never arrives,
// and waits for the barrier's first phase with the same bounded loop, under the
// caller's limit. No fault, trap or endless loop is involved.
#include <cstdint>
#include <cuda_runtime.h>

#include "dsa.h"
#include "ptx.cuh"

namespace dsa {

__global__ void __launch_bounds__(32) wait_probe_kernel(int* __restrict__ err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x != 0) return;
  // Phase 0 needs one arrival that never comes.
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(smem_u32(&bar), 0)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      record_error(err, kDevTimeout);
      return;
    }
  }
}

}  // namespace dsa

extern "C" dsa_status_t dsa_wait_probe(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return DSA_ERR_INVALID_ARG;
  if (!ws || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255) != 0) return DSA_ERR_WORKSPACE;
  dsa::wait_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(reinterpret_cast<int*>(ws),
                                                                            1000ull * limit_us);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
