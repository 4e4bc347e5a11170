// Radix top-k over fp32 score rows (the "radix top-k" of lmdeploy
// "feat: support GLM-5.2", Changes; negative-index padding per lmdeploy
// "glm5.3-flash support", Operator-level gains).
//
// One CTA of 1024 threads per row segment of at most 16384 entries, held in
// registers as runs of 4, 8 or 16 consecutive entries per thread (the smallest run
// that covers the segment, so that the row spreads over as many threads as it can;
// read as 16-byte loads where the row is aligned). Scores map to 32-bit keys whose
// unsigned order is the float order (-0 folded onto +0). A histogram of the top 11
// key bits locates the bin holding the k-th largest key; unless that bin is taken
// whole, its keys are copied to a shared-memory candidate list, and the next 11 and
// then 10 bits are resolved over that short list only. An element is then taken if
// its masked key is above the prefix so found, or equal to it and among the first
// `rem` equal ones by position (ties to the lower position). Output positions come
// from one block-wide exclusive scan of every thread's (above, equal) counts, in
// position order since each thread holds a contiguous run, so indices leave in
// ascending order.
//
// Rows longer than one CTA's capacity are split into chunks whose exact top-k
// (with their keys) become candidates; a second pass over the concatenated
// candidates, which are in ascending original position, gives the row's top-k.
// Any element of the row's top-k is in its chunk's top-k, so this is exact.
#include <cstdint>
#include "kernels.cuh"

namespace dsa {

constexpr int kTopkThreads = 1024;
constexpr int kTopkItems = 16;
constexpr int kTopkCapacity = kTopkThreads * kTopkItems;  // 16384

__device__ __forceinline__ uint32_t orderable_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkLaunch {
  GeomDev g;
  int k;
  int mode;                // 0: scores -> final idx; 1: scores chunk -> candidates; 2: candidates -> final idx
  const float* scores;     // modes 0, 1
  int64_t score_stride;
  int chunk;               // mode 1: chunk length; mode 2: unused
  int nchunks;             // mode 1: chunks per row; mode 2: candidate chunks per row (row len = nchunks*k)
  const uint32_t* cand_key_in;   // mode 2
  const int* cand_idx_in;        // mode 2
  uint32_t* cand_key_out;        // mode 1
  int* cand_idx_out;             // mode 1
  int* idx_out;                  // modes 0, 2: [T, k]
  int* err;
};

struct TopkShared {
  int hist[2048];
  int wsum[32];
  int sel_bin, sel_above, sel_cnt;
  int ncand;     // candidates appended so far
  int total;     // block total of the last scan
};

// Exclusive scan over the block of one int per thread (block total in *total).
__device__ __forceinline__ int topk_block_scan(int v, TopkShared& S, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) S.wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = S.wsum[lane];
    int iw = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, iw, o);
      if (lane >= o) iw += u;
    }
    S.wsum[lane] = iw - w;
    if (lane == 31) S.total = iw;
  }
  __syncthreads();
  if (total) *total = S.total;
  return S.wsum[warp] + incl - v;
}

// From the histogram S.hist[0..nb), highest bin first, find the bin holding the
// rem-th largest counted key: sel_bin, sel_above (count above it), sel_cnt. Thread t
// owns bins nb-1-2t and nb-2-2t.
__device__ __forceinline__ void topk_find_bin(TopkShared& S, int nb, int rem) {
  const int tid = threadIdx.x;
  const int hi_bin = nb - 1 - 2 * tid;
  const int c0 = hi_bin >= 0 ? S.hist[hi_bin] : 0;
  const int c1 = hi_bin - 1 >= 0 ? S.hist[hi_bin - 1] : 0;
  const int own = c0 + c1;
  const int excl = topk_block_scan(own, S, nullptr);
  if (own > 0 && excl < rem && rem <= excl + own) {
    if (excl + c0 >= rem) { S.sel_bin = hi_bin; S.sel_above = excl; S.sel_cnt = c0; }
    else { S.sel_bin = hi_bin - 1; S.sel_above = excl + c0; S.sel_cnt = c1; }
  }
  __syncthreads();
}

// The selection proper over a segment whose n (> k) entries are spread as runs of
// CNT per thread. cand: shared array of at least min(n, capacity) keys.
template <int CNT>
__device__ __forceinline__ void topk_select(const TopkLaunch& L, int n, int64_t in_base, int64_t out_base,
                                            int idx_offset, TopkShared& S, uint32_t* cand, int* out_s,
                                            uint32_t* key_s) {
  const int tid = threadIdx.x;
  const int k = L.k;
  const int e0 = tid * CNT;
  uint32_t key[CNT];
  uint32_t valid = 0;
  if (L.mode != 2 && e0 + CNT <= n && ((reinterpret_cast<uintptr_t>(L.scores + in_base) & 15) == 0)) {
    const float4* src = reinterpret_cast<const float4*>(L.scores + in_base + e0);
#pragma unroll
    for (int q = 0; q < CNT / 4; ++q) {
      const float4 v = src[q];
      key[4 * q] = orderable_key(v.x); key[4 * q + 1] = orderable_key(v.y);
      key[4 * q + 2] = orderable_key(v.z); key[4 * q + 3] = orderable_key(v.w);
    }
    valid = (CNT == 32) ? 0xffffffffu : ((1u << CNT) - 1u);
  } else {
#pragma unroll
    for (int i = 0; i < CNT; ++i) {
      const int e = e0 + i;
      key[i] = 0u;
      if (e < n) {
        if (L.mode == 2) {
          key[i] = L.cand_key_in[in_base + e];
          if (L.cand_idx_in[in_base + e] >= 0) valid |= 1u << i;
        } else {
          key[i] = orderable_key(L.scores[in_base + e]);
          valid |= 1u << i;
        }
      }
    }
  }

  // ---- pass over the top 11 bits (21-31) of every valid key
  for (int j = tid; j < 2048; j += kTopkThreads) S.hist[j] = 0;
  if (tid == 0) { S.sel_bin = 0; S.sel_above = 0; S.sel_cnt = -1; }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < CNT; ++i)
    if ((valid >> i) & 1u) atomicAdd(&S.hist[key[i] >> 21], 1);
  __syncthreads();
  topk_find_bin(S, 2048, k);
  int rem = k - S.sel_above;
  uint32_t prefix = (uint32_t)S.sel_bin << 21, pmask = 0xFFE00000u;
  if (S.sel_cnt != rem) {
    // ---- the keys of the threshold bin become a short candidate list; the lower
    // 21 bits are resolved over that list only (bits 10-20, then 0-9)
    const int ncand0 = S.sel_cnt;
    __syncthreads();   // every thread has read sel_* before they are reset
    if (tid == 0) S.ncand = 0;
    for (int j = tid; j < 2048; j += kTopkThreads) S.hist[j] = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < CNT; ++i) {
      if (((valid >> i) & 1u) && (key[i] & pmask) == prefix) {
        const int at = atomicAdd(&S.ncand, 1);
        cand[at] = key[i];
        atomicAdd(&S.hist[(key[i] >> 10) & 2047u], 1);
      }
    }
    if (tid == 0) { S.sel_bin = 0; S.sel_above = 0; S.sel_cnt = -1; }
    __syncthreads();
    topk_find_bin(S, 2048, rem);
    rem -= S.sel_above;
    prefix |= (uint32_t)S.sel_bin << 10;
    pmask |= 0x001FFC00u;
    if (S.sel_cnt != rem) {
      __syncthreads();
      for (int j = tid; j < 1024; j += kTopkThreads) S.hist[j] = 0;
      if (tid == 0) { S.sel_bin = 0; S.sel_above = 0; S.sel_cnt = -1; }
      __syncthreads();
      for (int c = tid; c < ncand0; c += kTopkThreads) {
        const uint32_t kc = cand[c];
        if ((kc & pmask) == prefix) atomicAdd(&S.hist[kc & 1023u], 1);
      }
      __syncthreads();
      topk_find_bin(S, 1024, rem);
      rem -= S.sel_above;
      prefix |= (uint32_t)S.sel_bin;
      pmask = 0xFFFFFFFFu;
    }
  }

  // ---- ordered placement: one block scan of (above << 16 | equal) counts (each
  // total <= 16384, so no carry); an element is taken if its masked key is above the
  // prefix, or equal and among the first `rem` equal ones by position
  uint32_t gt_bits = 0, eq_bits = 0;
#pragma unroll
  for (int i = 0; i < CNT; ++i) {
    const uint32_t m = key[i] & pmask;
    if (((valid >> i) & 1u) && m > prefix) gt_bits |= 1u << i;
    if (((valid >> i) & 1u) && m == prefix) eq_bits |= 1u << i;
  }
  const int excl = topk_block_scan((__popc(gt_bits) << 16) | __popc(eq_bits), S, nullptr);
  int rg = excl >> 16, re = excl & 0xffff;
  if (gt_bits | eq_bits) {
#pragma unroll
    for (int i = 0; i < CNT; ++i) {
      const bool is_gt = (gt_bits >> i) & 1u, is_eq = (eq_bits >> i) & 1u;
      if (is_gt || (is_eq && re < rem)) {
        const int pos = rg + min(re, rem);
        const int e = e0 + i;
        if (L.mode == 1) { out_s[pos] = idx_offset + e; key_s[pos] = key[i]; }
        else if (L.mode == 0) out_s[pos] = e;
        else out_s[pos] = L.cand_idx_in[in_base + e];
      }
      if (is_gt) ++rg;
      if (is_eq) ++re;
    }
  }
  __syncthreads();
  if (L.mode == 1) {
    for (int j = tid; j < k; j += kTopkThreads) {
      L.cand_idx_out[out_base + j] = out_s[j];
      L.cand_key_out[out_base + j] = key_s[j];
    }
  } else {
    for (int j = tid; j < k; j += kTopkThreads) L.idx_out[out_base + j] = out_s[j];
  }
}

__global__ void __launch_bounds__(kTopkThreads, 1) topk_kernel(const TopkLaunch L) {
  __shared__ TopkShared S;
  __shared__ int row_len_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int t, c = 0;
  if (L.mode == 1) { t = blockIdx.x / L.nchunks; c = blockIdx.x % L.nchunks; }
  else t = blockIdx.x;

  // Row length from the geometry (an input of the call, not of the preceding
  // kernel), found by one warp while the scores may still be in flight.
  if (warp == 0) {
    const QueryInfo qi = query_info_warp(L.g, t);
    if (lane == 0) {
      int n;
      if (L.mode == 2) {
        // A row with no more valid keys than k keeps all of them: its candidates are
        // exactly positions 0..pos, so it takes the short path below with n = pos+1.
        const int valid = qi.ok ? qi.pos + 1 : 0;
        n = valid <= L.k ? valid : L.nchunks * L.k;
      } else {
        if (!qi.ok) { record_error(L.err, kDevBadIndex); n = 0; }
        else n = qi.pos + 1;
        if (L.mode == 1) n = max(0, min(L.chunk, n - c * L.chunk));
      }
      row_len_s = n;
    }
  }
  griddep_launch_dependents();
  griddep_wait();   // scores (or candidates) come from the preceding kernel
  __syncthreads();
  const int n = row_len_s;
  const int k = L.k;

  // Where the row's entries and outputs live.
  const int64_t in_base = (L.mode == 0) ? (int64_t)t * L.score_stride
                        : (L.mode == 1) ? (int64_t)t * L.score_stride + (int64_t)c * L.chunk
                                        : (int64_t)t * L.nchunks * k;
  const int64_t out_base = (L.mode == 1) ? ((int64_t)t * L.nchunks + c) * k : (int64_t)t * k;
  const int idx_offset = (L.mode == 1) ? c * L.chunk : 0;

  if (n <= k) {
    // Everything valid is taken; positions are already ascending.
    for (int i = tid; i < k; i += kTopkThreads) {
      if (L.mode == 1) {
        const bool v = i < n;
        L.cand_key_out[out_base + i] = v ? orderable_key(L.scores[in_base + i]) : 0u;
        L.cand_idx_out[out_base + i] = v ? idx_offset + i : -1;
      } else if (L.mode == 0) {
        L.idx_out[out_base + i] = i < n ? i : -1;
      } else {  // mode 2: the first chunk's candidates are positions 0..n-1 in order
        L.idx_out[out_base + i] = i < n ? L.cand_idx_in[in_base + i] : -1;
      }
    }
    return;
  }
  // Dynamic shared memory: [k] staged output indices, [k] keys (mode 1), then the
  // candidate list of the threshold bin (at most n <= capacity keys).
  extern __shared__ int dyn_s[];
  int* out_s = dyn_s;
  uint32_t* key_s = reinterpret_cast<uint32_t*>(out_s + k);
  uint32_t* cand = key_s + (L.mode == 1 ? k : 0);
  // runs of 4, 8 or 16 entries per thread, whichever spreads the row over the most threads
  if (n <= 4 * kTopkThreads) topk_select<4>(L, n, in_base, out_base, idx_offset, S, cand, out_s, key_s);
  else if (n <= 8 * kTopkThreads) topk_select<8>(L, n, in_base, out_base, idx_offset, S, cand, out_s, key_s);
  else topk_select<16>(L, n, in_base, out_base, idx_offset, S, cand, out_s, key_s);
}

// Host-side launch sequence (called from the API layer). Returns a cudaError_t.
struct TopkPlan {
  int levels;      // 1: direct; 2: chunks + merge
  int chunk;
  int nchunks;
};

TopkPlan topk_plan(int max_seq_len, int k) {
  TopkPlan p;
  if (max_seq_len <= kTopkCapacity) { p.levels = 1; p.chunk = 0; p.nchunks = 1; return p; }
  p.levels = 2;
  p.chunk = kTopkCapacity;
  p.nchunks = (max_seq_len + kTopkCapacity - 1) / kTopkCapacity;
  return p;
}

size_t topk_workspace_bytes(int T, int max_seq_len, int k) {
  const TopkPlan p = topk_plan(max_seq_len, k);
  if (p.levels == 1) return 0;
  return (size_t)T * p.nchunks * k * (sizeof(uint32_t) + sizeof(int));
}

// Dynamic shared memory of one launch: the staged outputs (indices, and keys in mode
// 1) and the candidate keys of the threshold bin (at most one row segment's entries).
static size_t topk_smem_bytes(const TopkLaunch& L, int seg_len) {
  return (size_t)L.k * (L.mode == 1 ? 8 : 4) + (size_t)seg_len * 4;
}

static cudaError_t launch_topk_kernel(const TopkLaunch& L, int grid, int seg_len, bool pdl, cudaStream_t st) {
  const size_t smem = topk_smem_bytes(L, seg_len);
  // the 48 KB default covers static and dynamic shared memory together
  if (smem + sizeof(TopkShared) + 64 > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // The attention kernel that follows needs the whole shared-memory carveout; an SM
  // left in the same configuration takes its CTAs without reconfiguring.
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kTopkThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at; cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel, L);
}

cudaError_t topk_launch(const GeomDev& g, const float* scores, int64_t stride, int k, int* idx,
                        void* scratch, int* err, bool pdl, cudaStream_t st) {
  const TopkPlan p = topk_plan(g.max_seq_len, k);
  TopkLaunch L{};
  L.g = g; L.k = k; L.scores = scores; L.score_stride = stride; L.idx_out = idx; L.err = err;
  if (p.levels == 1) {
    L.mode = 0;
    return launch_topk_kernel(L, g.T, g.max_seq_len, pdl, st);
  }
  uint32_t* ck = reinterpret_cast<uint32_t*>(scratch);
  int* ci = reinterpret_cast<int*>(ck + (size_t)g.T * p.nchunks * k);
  L.mode = 1; L.chunk = p.chunk; L.nchunks = p.nchunks; L.cand_key_out = ck; L.cand_idx_out = ci;
  cudaError_t e = launch_topk_kernel(L, g.T * p.nchunks, p.chunk, pdl, st);
  if (e != cudaSuccess) return e;
  L.mode = 2; L.cand_key_in = ck; L.cand_idx_in = ci;
  return launch_topk_kernel(L, g.T, p.nchunks * k, true, st);   // follows the chunk pass just launched
}

}  // namespace dsa
