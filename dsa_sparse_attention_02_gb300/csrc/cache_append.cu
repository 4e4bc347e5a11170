// Cache append: the new tokens' latent rows and index keys written into the paged
// caches (lmdeploy "feat: support GLM-5.2", Changes: BF16/FP8 sparse FlashMLA cache
// paths and the MLA cache dtype policy; lmdeploy "glm5.3-flash support": cache
// updates run on every draft step).
//
// New token j of request b (flattened like the queries) is the request's position
// L_b - n_b + j, physical row block_table[b][pos / 64] * 64 + pos % 64 -- the rows
// the indexer and the attention read for it. One warp per token:
//   * bf16 latent cache: the 1152-byte row copied as given;
//   * int8 latent record (mlx-lm "GLM-5.2 (glm_moe_dsa) inference": int8 MLA latent
//     KV): as the e4m3 record with scale = amax / 127 and codes rounded to the
//     nearest integer (ties to even), clamped to +-127;
//   * e4m3 latent record (656 B): lane l quantizes latent values 16l..16l+15; the
//     eight lanes of a 128-value group reduce its amax, scale = amax / 448 (1 for an
//     all-zero group), code = e4m3(x / scale) with the quotient in fp32 and the
//     conversion rounding to nearest even and saturating at +-448; the 512 codes, the
//     four scales and the 64 RoPE values as given (bf16) go to the token's slot of
//     its page's code, scale and RoPE planes;
//   * index key: e4m3 with one such scale per token over its 128 values (the scale to
//     the [P, 64] tensor), or the bf16 key as given.
// Every row other than the new tokens' is left as it was. Page ids out of range
// skip the token and report DSA_ERR_BAD_INDEX.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include "kernels.cuh"

namespace dsa {

constexpr int kAppendWarps = 4;
constexpr float kE4m3Max = 448.f;
constexpr float kI8Max = 127.f;

// Four e4m3 codes (byte i from value i): round to nearest even, saturate at +-448.
__device__ __forceinline__ uint32_t e4m3_pack4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

// Four int8 codes (byte i from value i): round to nearest even, clamp to +-127.
__device__ __forceinline__ uint32_t i8_pack4(float a, float b, float c, float d) {
  const float f[4] = {a, b, c, d};
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = max(-127, min(127, __float2int_rn(f[i])));
    r |= (uint32_t)(q & 0xFF) << (8 * i);
  }
  return r;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(32 * kAppendWarps) cache_append_kernel(const AppendArgs A) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kAppendWarps + warp;
  if (t >= A.g.T) return;
  // The token's data does not depend on where it goes: its loads are issued before
  // the row lookup (request search, block table), so the two latencies overlap.
  const uint4* src = reinterpret_cast<const uint4*>(A.kv_new) + (int64_t)t * 72;   // 576 bf16 = 72 x 16 B
  uint4 d0 = make_uint4(0, 0, 0, 0), d1 = d0, d2 = d0;
  const bool record = A.kv_format != kKvBf16;
  if (!record) {
    d0 = __ldg(src + lane);
    d1 = __ldg(src + 32 + lane);
    if (lane < 8) d2 = __ldg(src + 64 + lane);
  } else {
    d0 = __ldg(src + 2 * lane);
    d1 = __ldg(src + 2 * lane + 1);
    if (lane < 8) d2 = __ldg(src + 64 + lane);     // RoPE
  }
  uint2 kk = make_uint2(0, 0);
  if (A.k_new) kk = __ldg(reinterpret_cast<const uint2*>(A.k_new) + (int64_t)t * 32 + lane);   // 128 bf16

  const QueryInfo qi = query_info_warp(A.g, t);
  const int64_t row = qi.ok ? physical_row(A.g, qi.b, qi.pos) : -1;
  if (row < 0) {
    if (lane == 0) record_error(A.err, kDevBadIndex);
    return;
  }
  // ---- latent row
  if (!record) {
    uint4* dst = reinterpret_cast<uint4*>(A.kv_cache + row * (kDimQK * 2));
    dst[lane] = d0;
    dst[32 + lane] = d1;
    if (lane < 8) dst[64 + lane] = d2;
  } else {
    uint8_t* const kv = A.kv_cache;
    float v[16];
    {
      float a[8], b[8];
      bf16x8_to_f32(d0, a);
      bf16x8_to_f32(d1, b);
#pragma unroll
      for (int i = 0; i < 8; ++i) { v[i] = a[i]; v[8 + i] = b[i]; }
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));   // amax of the lane's 128-value group
    const bool i8 = A.kv_format == kKvInt8;
    const float scale = m > 0.f ? m / (i8 ? kI8Max : kE4m3Max) : 1.f;
    uint4 codes;
    auto pack4 = [&](int i) {
      const float a = v[i] / scale, b = v[i + 1] / scale, c = v[i + 2] / scale, d = v[i + 3] / scale;
      return i8 ? i8_pack4(a, b, c, d) : e4m3_pack4(a, b, c, d);
    };
    codes.x = pack4(0);
    codes.y = pack4(4);
    codes.z = pack4(8);
    codes.w = pack4(12);
    *reinterpret_cast<uint4*>(kv + rec_codes_at(row) + 16 * lane) = codes;
    if ((lane & 7) == 0) *reinterpret_cast<float*>(kv + rec_scales_at(row) + 4 * (lane >> 3)) = scale;
    if (lane < 8) *reinterpret_cast<uint4*>(kv + rec_rope_at(row) + 16 * lane) = d2;
  }
  // ---- index key
  if (A.k_new) {
    if (!A.k_fp8) {
      reinterpret_cast<uint2*>(A.k_cache + row * (kDimIdx * 2))[lane] = kk;
    } else {
      const float f0 = __uint_as_float(kk.x << 16), f1 = __uint_as_float(kk.x & 0xFFFF0000u);
      const float f2 = __uint_as_float(kk.y << 16), f3 = __uint_as_float(kk.y & 0xFFFF0000u);
      float m = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const float scale = m > 0.f ? m / kE4m3Max : 1.f;
      reinterpret_cast<uint32_t*>(A.k_cache + row * kDimIdx)[lane] =
          e4m3_pack4(f0 / scale, f1 / scale, f2 / scale, f3 / scale);
      if (lane == 0) A.k_scale[row] = scale;
    }
  }
}

cudaError_t cache_append_launch(const AppendArgs& A, cudaStream_t st) {
  const int grid = (A.g.T + kAppendWarps - 1) / kAppendWarps;
  cache_append_kernel<<<grid, 32 * kAppendWarps, 0, st>>>(A);
  return cudaGetLastError();
}

}  // namespace dsa
