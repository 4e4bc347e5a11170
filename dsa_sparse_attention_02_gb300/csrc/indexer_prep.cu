// Indexer query/key preparation, fused: RoPE on the indexer queries and keys,
// LayerNorm on the keys, e4m3 quantization of both, and the key's write into the
// paged index cache (lmdeploy "feat: support GLM-5.2", Changes: fused indexer
// preparation in the DSA indexing work; Performance: fused Q/K preprocessing of the
// indexer; mlx-lm "GLM-5.2 (glm_moe_dsa) inference", Changes: the indexer's RoPE is
// non-interleaved and its LayerNorm eps is 1e-6).
//
// For query token t (flattened like the queries) at position pos(t):
//   q_out[t,h,:] = e4m3(RoPE(q_in[t,h,:]) / s),  q_scale[t,h] = s = amax / 448
//   key row of pos(t):  e4m3(RoPE(LayerNorm(k_in[t,:])) / s_k), scale s_k
// RoPE is non-interleaved on the first rope_dim values: for i < r = rope_dim/2,
//   y_i = x_i cos - x_{i+r} sin,  y_{i+r} = x_{i+r} cos + x_i sin,
// with cos/sin read from [max_seq_len, r] tables at pos(t); the rest pass through.
// LayerNorm: (x - mean) / sqrt(var + eps) * gamma + beta, biased variance. All in
// fp32 from the bf16 inputs; the scale and the quotient are IEEE fp32 divisions and
// the code is the nearest e4m3 value (ties to even), saturating at +-448; an
// all-zero vector gets scale 1.
//
// One block per token: its query rows and key arrive in shared memory by bulk copy;
// a warp prepares four query heads at a time (their stages run together so that the
// dependent shuffle chains overlap), one warp the key; lane l holds values 4l..4l+3
// of each vector. The RoPE partner of lane l < r/4 is lane l + r/4 (and
// back), fetched by one shuffle per value. A token whose geometry is inconsistent,
// or whose key page is out of range, is skipped and reported (DSA_ERR_BAD_INDEX).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include "kernels.cuh"

namespace dsa {

constexpr int kPrepWarps = 8;            // warps per block (one block per token)
constexpr int kPrepG = 4;                // query heads per warp, processed stage by stage together
constexpr float kPrepE4m3Max = 448.f;

__device__ __forceinline__ uint32_t prep_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

__device__ __forceinline__ void bf16x4(uint2 r, float* x) {
  x[0] = __uint_as_float(r.x << 16);
  x[1] = __uint_as_float(r.x & 0xFFFF0000u);
  x[2] = __uint_as_float(r.y << 16);
  x[3] = __uint_as_float(r.y & 0xFFFF0000u);
}

// Non-interleaved RoPE of N vectors of 128 values (4 per lane): lane l < hl holds
// first-half values, lane hl <= l < 2hl the second half (hl = rope_dim/8); c, s are
// this token's cos/sin for the lane's four pairs.
template <int N>
__device__ __forceinline__ void prep_rope(float (&x)[N][4], int hl, int lane, const float (&c)[4], const float (&s)[4]) {
  const bool first = lane < hl, second = lane >= hl && lane < 2 * hl;
  const int src = first ? lane + hl : (second ? lane - hl : lane);
  float o[N][4];
#pragma unroll
  for (int g = 0; g < N; ++g)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[g][j] = __shfl_sync(0xffffffffu, x[g][j], src);
  const float sg = first ? -1.f : 1.f;   // y_i = x_i c - x_{i+r} s; y_{i+r} = x_{i+r} c + x_i s
  if (first || second) {
#pragma unroll
    for (int g = 0; g < N; ++g)
#pragma unroll
      for (int j = 0; j < 4; ++j) x[g][j] = x[g][j] * c[j] + sg * (o[g][j] * s[j]);
  }
}

// Scales (amax / 448, 1 for all zero) of N vectors and this lane's four codes of each.
// The amax is one warp reduction of the magnitudes' bit patterns, which order like
// the magnitudes themselves (non-negative, finite).
template <int N>
__device__ __forceinline__ void prep_quantize(const float (&x)[N][4], float (&scale)[N], uint32_t (&codes)[N]) {
  float m[N];
#pragma unroll
  for (int g = 0; g < N; ++g) {
    const float lm = fmaxf(fmaxf(fabsf(x[g][0]), fabsf(x[g][1])), fmaxf(fabsf(x[g][2]), fabsf(x[g][3])));
    m[g] = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(lm)));
  }
#pragma unroll
  for (int g = 0; g < N; ++g) {
    scale[g] = m[g] > 0.f ? m[g] / kPrepE4m3Max : 1.f;
    codes[g] = prep_e4m3x4(x[g][0] / scale[g], x[g][1] / scale[g], x[g][2] / scale[g], x[g][3] / scale[g]);
  }
}

// Blocks split x tokens: block (t, part) takes 4-head groups [g0, g1) of token t,
// the last part also its key. Thread 0 brings those query rows and the key into
// shared memory with bulk copies (one mbarrier); meanwhile every warp looks up the
// token's position and its cos/sin row, and the key's warp the cache row. Then warp
// w prepares groups g0 + w, g0 + w + 8, ... (four heads each, their stages run
// together), and the warp after the last group the key.
__global__ void __launch_bounds__(32 * kPrepWarps) indexer_prep_kernel(const PrepArgs A) {
  extern __shared__ __align__(128) uint8_t prep_smem[];   // [Hi][256 B] queries, then the key's 256 B
  __shared__ uint64_t full_bar;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x / A.split, part = blockIdx.x - t * A.split;
  const int groups = (A.Hi + kPrepG - 1) / kPrepG;
  const int g0 = part * groups / A.split, g1 = (part + 1) * groups / A.split;
  const int h_begin = g0 * kPrepG, h_end = min(g1 * kPrepG, A.Hi);
  const bool has_key = A.k_in != nullptr && part == A.split - 1;
  const uint32_t qbytes = (uint32_t)(h_end - h_begin) * 256u;
  const uint32_t bar = smem_u32(&full_bar);
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, qbytes + (has_key ? 256u : 0u));
    bulk_load(smem_u32(prep_smem), reinterpret_cast<const uint8_t*>(A.q_in) + ((int64_t)t * A.Hi + h_begin) * 256,
              qbytes, bar);
    if (has_key) bulk_load(smem_u32(prep_smem + qbytes), reinterpret_cast<const uint8_t*>(A.k_in) + (int64_t)t * 256, 256u, bar);
  }
  __syncthreads();   // the barrier is initialized before anyone waits on it
  const bool key_warp = has_key && warp == (g1 - g0) % kPrepWarps;
  const QueryInfo qi = query_info_warp(A.g, t);
  const int64_t krow = (key_warp && qi.ok) ? physical_row(A.g, qi.b, qi.pos) : -1;
  const int r = A.rope_dim >> 1, hl = r >> 2;
  float c[4] = {1.f, 1.f, 1.f, 1.f}, sn[4] = {0.f, 0.f, 0.f, 0.f};
  if (qi.ok && lane < 2 * hl) {
    const int i0 = 4 * (lane < hl ? lane : lane - hl);
    const float4 cv = *reinterpret_cast<const float4*>(A.rope_cos + (int64_t)qi.pos * r + i0);
    const float4 sv = *reinterpret_cast<const float4*>(A.rope_sin + (int64_t)qi.pos * r + i0);
    c[0] = cv.x; c[1] = cv.y; c[2] = cv.z; c[3] = cv.w;
    sn[0] = sv.x; sn[1] = sv.y; sn[2] = sv.z; sn[3] = sv.w;
  }
  // every thread waits for the copies (the block must not exit with them in flight)
  if (!mbar_wait(bar, 0, &abort_flag, A.err)) return;
  if (!qi.ok) {
    if (tid == 0) record_error(A.err, kDevBadIndex);
    return;
  }
  for (int grp = g0 + warp; grp < g1; grp += kPrepWarps) {
    const int h0 = grp * kPrepG;
    float x[kPrepG][4];
#pragma unroll
    for (int g = 0; g < kPrepG; ++g) {
      const int h = min(h0 + g, h_end - 1);
      bf16x4(*reinterpret_cast<const uint2*>(prep_smem + (h - h_begin) * 256 + lane * 8), x[g]);
    }
    prep_rope<kPrepG>(x, hl, lane, c, sn);
    float scale[kPrepG];
    uint32_t codes[kPrepG];
    prep_quantize<kPrepG>(x, scale, codes);
#pragma unroll
    for (int g = 0; g < kPrepG; ++g) {
      if (h0 + g < A.Hi) {
        reinterpret_cast<uint32_t*>(A.q_out)[((int64_t)t * A.Hi + h0 + g) * 32 + lane] = codes[g];
        if (lane == 0) A.q_scale[(int64_t)t * A.Hi + h0 + g] = scale[g];
      }
    }
  }
  if (!key_warp) return;
  float x[1][4];
  bf16x4(*reinterpret_cast<const uint2*>(prep_smem + qbytes + lane * 8), x[0]);
  const float mean = warp_sum((x[0][0] + x[0][1]) + (x[0][2] + x[0][3])) * (1.f / 128.f);
  float d[4], v = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) { d[q] = x[0][q] - mean; v = fmaf(d[q], d[q], v); }
  const float var = warp_sum(v) * (1.f / 128.f);
  const float rstd = 1.f / sqrtf(var + A.ln_eps);
  float4 gm = make_float4(1.f, 1.f, 1.f, 1.f), bt = make_float4(0.f, 0.f, 0.f, 0.f);
  if (A.ln_gamma) gm = *reinterpret_cast<const float4*>(A.ln_gamma + 4 * lane);
  if (A.ln_beta) bt = *reinterpret_cast<const float4*>(A.ln_beta + 4 * lane);
  x[0][0] = fmaf(d[0] * rstd, gm.x, bt.x);
  x[0][1] = fmaf(d[1] * rstd, gm.y, bt.y);
  x[0][2] = fmaf(d[2] * rstd, gm.z, bt.z);
  x[0][3] = fmaf(d[3] * rstd, gm.w, bt.w);
  prep_rope<1>(x, hl, lane, c, sn);
  float scale[1];
  uint32_t codes[1];
  prep_quantize<1>(x, scale, codes);
  if (krow < 0) {
    if (lane == 0) record_error(A.err, kDevBadIndex);
    return;
  }
  reinterpret_cast<uint32_t*>(A.k_cache + krow * kDimIdx)[lane] = codes[0];
  if (lane == 0) A.k_scale[krow] = scale[0];
}

cudaError_t indexer_prep_launch(const PrepArgs& A, cudaStream_t st) {
  // the largest part's query rows (whole groups, at most Hi) and the key: <= 33 KB,
  // within the default 48 KB
  const int groups = (A.Hi + kPrepG - 1) / kPrepG;
  const int max_groups = (groups + A.split - 1) / A.split;
  const size_t smem = (size_t)(max_groups * kPrepG < A.Hi ? max_groups * kPrepG : A.Hi) * 256 + 256;
  indexer_prep_kernel<<<(unsigned)((int64_t)A.g.T * A.split), 32 * kPrepWarps, smem, st>>>(A);
  return cudaGetLastError();
}

}  // namespace dsa
