// Geometry shared by the kernels: flattened varlen queries over paged caches.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include "ptx.cuh"

namespace dsa {

constexpr int kPage = 64;
constexpr int kDimIdx = 128;      // indexer head dim
constexpr int kDimLatent = 512;   // latent (value) width
constexpr int kDimRope = 64;
constexpr int kDimQK = 576;       // 512 latent + 64 RoPE
constexpr int kFp8Record = 656;   // latent record bytes per token (e4m3 or int8 codes)
// A page of latent records holds its 64 tokens' fields as three planes: codes
// [64][512], fp32 scales [64][4], bf16 RoPE [64][64]; every token's codes start on a
// 512-byte boundary and its RoPE values on a 128-byte one.
constexpr int kRecPageBytes = kPage * kFp8Record;                   // 41984
constexpr int kRecScalesAt = kPage * kDimLatent;                    // 32768
constexpr int kRecRopeAt = kRecScalesAt + kPage * 16;               // 33792

// Radix keys of the top-k: a 32-bit key whose unsigned order is the order of the
// fp32 scores (-0 folded onto +0). The top-k's first digit is the key's top 11 bits;
// the fused step's indexer counts them per row and per 16384-position chunk
// (first-digit histograms of kHistBins ints), which the top-k then reads instead of
// counting them itself.
__device__ __forceinline__ uint32_t orderable_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
constexpr int kHistBins = 2048;
constexpr int kHistShift = 21;          // bin = key >> 21
constexpr int kTopkChunkLog2 = 14;      // top-k chunks of 16384 positions
// Word of the workspace header (after the error word) that counts the segments whose
// first-digit histogram the top-k rejected.
constexpr int kHistRejectedWord = 1;

struct GeomDev {
  int B, T, max_seq_len, num_pages, bt_stride;
  const int* seq_lens;
  const int* cu_q;
  const int* block_table;
};

// Request of flattened query t: the largest b with cu_q[b] <= t (binary search).
__device__ __forceinline__ int query_request(const GeomDev& g, int t) {
  int lo = 0, hi = g.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(g.cu_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct QueryInfo {
  int b;      // request
  int pos;    // causal position; keys 0..pos are visible
  int len;    // seq_lens[b]
  bool ok;    // geometry consistent
};

__device__ __forceinline__ QueryInfo query_info(const GeomDev& g, int t) {
  QueryInfo qi;
  qi.b = query_request(g, t);
  const int q0 = __ldg(g.cu_q + qi.b), q1 = __ldg(g.cu_q + qi.b + 1);
  qi.len = __ldg(g.seq_lens + qi.b);
  qi.pos = qi.len - (q1 - q0) + (t - q0);
  qi.ok = (t >= q0) && (t < q1) && (qi.len <= g.max_seq_len) && (qi.pos >= 0) &&
          (qi.pos < qi.len);
  return qi;
}

// query_info computed by a whole warp: the request search probes 32 entries of
// cu_q per round (one round for B <= 32, two for B <= 1024) instead of a serial
// binary search. Every lane returns the same result.
__device__ __forceinline__ QueryInfo query_info_warp(const GeomDev& g, int t) {
  const int lane = threadIdx.x & 31;
  int lo = 0, n = g.B;                       // answer in [lo, lo + n)
  while (n > 32) {
    const int step = (n + 31) / 32;
    const int idx = lo + lane * step;
    const bool le = idx < lo + n && __ldg(g.cu_q + idx) <= t;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    const int last = m ? 31 - __clz(m) : 0;
    lo += last * step;
    n = min(step, n - last * step);
  }
  const int idx = lo + lane;
  const bool le = lane < n && __ldg(g.cu_q + idx) <= t;
  const unsigned m = __ballot_sync(0xffffffffu, le);
  QueryInfo qi;
  qi.b = lo + (m ? 31 - __clz(m) : 0);
  const int q0 = __ldg(g.cu_q + qi.b), q1 = __ldg(g.cu_q + qi.b + 1);
  qi.len = __ldg(g.seq_lens + qi.b);
  qi.pos = qi.len - (q1 - q0) + (t - q0);
  qi.ok = (t >= q0) && (t < q1) && (qi.len <= g.max_seq_len) && (qi.pos >= 0) && (qi.pos < qi.len);
  return qi;
}

// Byte offsets of physical row r's fields in a latent record cache.
__host__ __device__ __forceinline__ int64_t rec_codes_at(int64_t r) {
  return (r >> 6) * kRecPageBytes + (r & 63) * kDimLatent;
}
__host__ __device__ __forceinline__ int64_t rec_scales_at(int64_t r) {
  return (r >> 6) * kRecPageBytes + kRecScalesAt + (r & 63) * 16;
}
__host__ __device__ __forceinline__ int64_t rec_rope_at(int64_t r) {
  return (r >> 6) * kRecPageBytes + kRecRopeAt + (r & 63) * (kDimRope * 2);
}

// Physical row (page*64 + s%64) of request b's logical token s, or -1 if the page id
// is out of range.
__device__ __forceinline__ int64_t physical_row(const GeomDev& g, int b, int s) {
  const int page = __ldg(g.block_table + (int64_t)b * g.bt_stride + (s >> 6));
  if (page < 0 || page >= g.num_pages) return -1;
  return (int64_t)page * kPage + (s & 63);
}

// Static balanced split of `n` work items over `g` CTAs: CTA c owns
// [floor(c*n/g), floor((c+1)*n/g)). owner(x) is the CTA holding item x.
__host__ __device__ __forceinline__ int64_t split_begin(int64_t c, int64_t n, int64_t g) {
  return (c * n) / g;
}
__host__ __device__ __forceinline__ int64_t split_owner(int64_t x, int64_t n, int64_t g) {
  return ((x + 1) * g - 1) / n;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Named barrier among `count` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace dsa
