// dsa_stage_copy: a byte copy done by the SMs, for moving a step's packed inputs and
// outputs between page-locked host memory and the device. On a part whose host
// memory is reached over a coherent chip-to-chip link, SM loads and stores of
// page-locked host memory move data faster than a copy-engine transfer of the same
// size, and the copy is an ordinary kernel in the stream.
//
// Both pointers must be device memory or page-locked host memory that the device
// maps (cudaHostAlloc / cudaHostRegister); the host function resolves each through
// cudaPointerGetAttributes and refuses anything else before launching, so the
// kernel only ever touches addresses the device has mapped.
#include <cstdint>
#include "kernels.cuh"

namespace dsa {

constexpr int kStageThreads = 512;
constexpr int kStageUnroll = 4;

__global__ void __launch_bounds__(kStageThreads) stage_copy_kernel(uint4* __restrict__ dst,
                                                                   const uint4* __restrict__ src, size_t n16,
                                                                   uint8_t* __restrict__ dst_tail,
                                                                   const uint8_t* __restrict__ src_tail, int tail) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (kStageUnroll - 1) * stride < n16; i += kStageUnroll * stride) {
    uint4 v[kStageUnroll];
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) dst[i + u * stride] = v[u];
  }
  for (; i < n16; i += stride) dst[i] = src[i];
  if (blockIdx.x == 0 && (int)threadIdx.x < tail) dst_tail[threadIdx.x] = src_tail[threadIdx.x];
}

cudaError_t stage_copy_launch(void* dst, const void* src, size_t bytes, int num_sms, cudaStream_t st) {
  const size_t n16 = bytes / 16;
  const int tail = (int)(bytes - n16 * 16);
  size_t blocks = (n16 + (size_t)kStageThreads * kStageUnroll - 1) / ((size_t)kStageThreads * kStageUnroll);
  const size_t cap = (size_t)2 * (num_sms > 0 ? num_sms : 1);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  stage_copy_kernel<<<(unsigned)blocks, kStageThreads, 0, st>>>(
      reinterpret_cast<uint4*>(dst), reinterpret_cast<const uint4*>(src), n16,
      reinterpret_cast<uint8_t*>(dst) + n16 * 16, reinterpret_cast<const uint8_t*>(src) + n16 * 16, tail);
  return cudaGetLastError();
}

}  // namespace dsa
