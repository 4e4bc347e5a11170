// Radix top-k over fp32 score rows (the "radix top-k" of lmdeploy
// "feat: support GLM-5.2", Changes; negative-index padding per lmdeploy
// "glm5.3-flash support", Operator-level gains).
//
// One CTA of 1024 threads per row segment of at most 16384 entries, held in
// registers as runs of 4, 8 or 16 consecutive entries per thread (the smallest run
// that covers the segment, so that the row spreads over as many threads as it can;
// read as 16-byte loads where the row is aligned). Scores map to 32-bit keys whose
// unsigned order is the float order (-0 folded onto +0). Radix digits of up to 11
// bits, starting below the leading bits that every valid key shares, are resolved
// one after the other: a shared-memory histogram of the digit over the keys that
// match the prefix found so far (read from the registers each time) locates the bin
// holding the rem-th largest of them. Every warp finds that bin itself from the
// histogram, so a digit costs two block barriers. An element is then taken if its
// masked key is above the prefix so found, or equal to it and among the first `rem`
// equal ones by position (ties to the lower position). Output positions come from
// one block-wide exclusive scan of every thread's (above, equal) counts, in position
// order since each thread holds a contiguous run, so indices leave in ascending
// order; each thread writes its results straight to the output. A segment with no
// more valid entries than k keeps all of them.
//
// Rows longer than one CTA's capacity are cut into chunks of 16384 positions whose
// exact top-k (with their keys) become candidate lists. Lists are then merged in
// groups of min(4, floor(16384 / k)), level after level, until one list remains: a group's
// lists are concatenated in chunk order, so its candidates stay in ascending
// position and ties still go to the lower position. Any element of the row's top-k
// is in the top-k of every group that contains it, so every level is exact.
//
// Seeded instantiations (dsa_decode_step_hist) take the first digit's histogram (the
// keys' top 11 bits) from the indexer instead of counting it: the digits then start
// at the top bit, the selection is checked against the exact totals of its placement
// scan, and a segment whose histogram does not match its scores is selected again
// unseeded.
#include <cstdint>
#include "kernels.cuh"

namespace dsa {

constexpr int kTopkThreads = 1024;
constexpr int kTopkItems = 16;
constexpr int kTopkCapacity = kTopkThreads * kTopkItems;  // 16384
static_assert(kTopkCapacity == 1 << kTopkChunkLog2, "chunk length");
static_assert(kHistBins == 2 * kTopkThreads, "two first-digit bins per thread");

// Modes of one launch:
//   kDirect: score rows (<= 16384 long) -> final idx
//   kChunks: chunks c0 .. c0+nl-1 of every row -> candidate lists (key, position)
//   kMerge:  groups of `fan` candidate lists -> lists (n_out > 1) or final idx (n_out == 1)
enum : int { kDirect = 0, kChunks = 1, kMerge = 2 };

struct TopkLaunch {
  GeomDev g;
  int k;
  int mode;
  const float* scores;           // kDirect, kChunks (key c0*chunk of each row for kChunks)
  int64_t score_stride;
  int chunk;                     // kChunks: chunk length
  int c0, nl;                    // kChunks: first chunk of the launch, chunks per row in it
  int nchunks;                   // kChunks: chunks per row (layout of the candidate lists)
  int n_in, fan, n_out;          // kMerge: lists per row in, lists merged per group, lists per row out
  const uint32_t* cand_key_in;   // kMerge
  const int* cand_idx_in;        // kMerge
  uint32_t* cand_key_out;        // kChunks, kMerge with n_out > 1
  int* cand_idx_out;
  int* idx_out;                  // kDirect, kMerge with n_out == 1: [T, k]
  int* hist;                     // kDirect, kChunks: first-digit histograms [T][hist_chunks][2048], or null
  int hist_chunks;
  int* err;
};

struct TopkShared {
  int hist[2][2048];            // digit histograms (alternating between digits)
  int wsum[32];                 // per warp: its histogram bins' total
  int wscan[32];                // per warp: its placement counts
  uint32_t wand[32], wor[32];   // per warp: AND and OR of its valid keys
  int wcnt[32];                 // per warp: valid keys
};
constexpr int kTopkWarps = kTopkThreads / 32;
static_assert(kTopkWarps == 32 && 64 * kTopkWarps == 2048, "two bins per thread");

struct TopkBin { int bin, above, cnt; };

// The bin of histogram h[0..nb) that holds the rem-th largest counted key, with the
// count of keys in the bins above it and in it. Warp w sums bins nb-1-64w down to
// nb-64-64w (two per lane); after a barrier every warp scans the 32 warp totals,
// picks the warp range that holds the rem-th key and scans that range's bins, so that
// all threads return the same bin with no further barrier. The histogram must be
// complete on entry (the first barrier). zero: an array of 2048 ints that every warp
// has finished reading (before the first barrier), cleared for a later digit; or null.
__device__ __forceinline__ TopkBin topk_find_bin(TopkShared& S, const int* h, int nb, int rem, int* zero) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();   // every count is in h
  if (zero) { zero[threadIdx.x] = 0; zero[threadIdx.x + kTopkThreads] = 0; }
  {
    const int hi = nb - 1 - 64 * warp - 2 * lane;
    const int own = (hi >= 0 ? h[hi] : 0) + (hi >= 1 ? h[hi - 1] : 0);
    const int tot = (int)__reduce_add_sync(0xffffffffu, (uint32_t)own);
    if (lane == 0) S.wsum[warp] = tot;
  }
  __syncthreads();
  const int v = S.wsum[lane];
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  TopkBin r{0, 0, -1};
  const unsigned mw = __ballot_sync(0xffffffffu, v > 0 && incl - v < rem && rem <= incl);
  if (mw == 0u) return r;   // fewer than rem keys counted (not reached by the callers)
  const int W = __ffs(mw) - 1;
  const int above_w = __shfl_sync(0xffffffffu, incl - v, W);
  const int hi = nb - 1 - 64 * W - 2 * lane;
  const int c0 = hi >= 0 ? h[hi] : 0, c1 = hi >= 1 ? h[hi - 1] : 0;
  const int own = c0 + c1;
  int in2 = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, in2, o);
    if (lane >= o) in2 += u;
  }
  const int ex2 = above_w + in2 - own;
  const unsigned ml = __ballot_sync(0xffffffffu, own > 0 && ex2 < rem && rem <= ex2 + own);
  const int L = __ffs(ml) - 1;   // the range's counts add up to above_w + v >= rem
  const int bin = __shfl_sync(0xffffffffu, hi, L), ex = __shfl_sync(0xffffffffu, ex2, L);
  const int a0 = __shfl_sync(0xffffffffu, c0, L), a1 = __shfl_sync(0xffffffffu, c1, L);
  if (ex + a0 >= rem) { r.bin = bin; r.above = ex; r.cnt = a0; }
  else { r.bin = bin - 1; r.above = ex + a0; r.cnt = a1; }
  return r;
}

// The selection proper over a segment of n (> k) entries spread as runs of CNT per
// thread; entries whose valid bit is clear take no part. pos_s (merges): shared array
// of n ints for the input candidates' positions. Writes min(k, valid entries) results
// then -1 padding. kSeeded: hrow holds the segment's first-digit histogram (below).
template <int CNT, int MODE, bool kSeeded>
__device__ __forceinline__ bool topk_select(const TopkLaunch& L, int n, int64_t in_base, int64_t out_base,
                                            int idx_offset, TopkShared& S, int* pos_s, const int* hrow) {
  const int tid = threadIdx.x;
  const int k = L.k;
  const int e0 = tid * CNT;
  uint32_t key[CNT];
  uint32_t valid = 0;
  // candidate keys and positions with 16-byte accesses where all three addresses allow
  // them (k a multiple of 4 makes them aligned; other k take the scalar loop)
  const bool vec_merge = MODE == kMerge && e0 + CNT <= n &&
                         ((reinterpret_cast<uintptr_t>(L.cand_key_in + in_base + e0) |
                           reinterpret_cast<uintptr_t>(L.cand_idx_in + in_base + e0) |
                           reinterpret_cast<uintptr_t>(pos_s + e0)) & 15) == 0;
  if (vec_merge) {
    // the positions go to this thread's slots of pos_s (read back only by this thread
    // when it places its results)
    const uint4* ks = reinterpret_cast<const uint4*>(L.cand_key_in + in_base + e0);
    const int4* is = reinterpret_cast<const int4*>(L.cand_idx_in + in_base + e0);
#pragma unroll
    for (int q = 0; q < CNT / 4; ++q) {
      const uint4 kv = ks[q];
      const int4 iv = is[q];
      key[4 * q] = kv.x; key[4 * q + 1] = kv.y; key[4 * q + 2] = kv.z; key[4 * q + 3] = kv.w;
      *reinterpret_cast<int4*>(pos_s + e0 + 4 * q) = iv;
      valid |= (iv.x >= 0 ? 1u : 0u) << (4 * q) | (iv.y >= 0 ? 1u : 0u) << (4 * q + 1) |
               (iv.z >= 0 ? 1u : 0u) << (4 * q + 2) | (iv.w >= 0 ? 1u : 0u) << (4 * q + 3);
    }
  } else if (MODE != kMerge && e0 + CNT <= n && ((reinterpret_cast<uintptr_t>(L.scores + in_base) & 15) == 0)) {
    const float4* src = reinterpret_cast<const float4*>(L.scores + in_base + e0);
#pragma unroll
    for (int q = 0; q < CNT / 4; ++q) {
      const float4 v = src[q];
      key[4 * q] = orderable_key(v.x); key[4 * q + 1] = orderable_key(v.y);
      key[4 * q + 2] = orderable_key(v.z); key[4 * q + 3] = orderable_key(v.w);
    }
    valid = (1u << CNT) - 1u;
  } else {
#pragma unroll
    for (int i = 0; i < CNT; ++i) {
      const int e = e0 + i;
      key[i] = 0u;
      if (e < n) {
        if (MODE == kMerge) {
          key[i] = L.cand_key_in[in_base + e];
          const int ci = L.cand_idx_in[in_base + e];
          pos_s[e] = ci;
          if (ci >= 0) valid |= 1u << i;
        } else {
          key[i] = orderable_key(L.scores[in_base + e]);
          valid |= 1u << i;
        }
      }
    }
  }

  const int lane = tid & 31, warp = tid >> 5;
  int rem, count, incl, wincl, wv, packed;
  uint32_t prefix, pmask, gt_bits, eq_bits;
  // seeded: the first digit's histogram (the top 11 bits of every entry's key) comes
  // from the indexer, read while the entries are still in flight, and the digits start
  // at the top bit. The selection is then checked against its exact final counts; if
  // they disagree (a histogram that does not belong to these scores) nothing is
  // written and false is returned, for the caller to select again without it.
  constexpr bool seeded = MODE != kMerge && kSeeded;
  {
    int nvalid, consumed = 0;
    prefix = 0u; pmask = 0u;
    if constexpr (seeded) {
      const int2 h2 = reinterpret_cast<const int2*>(hrow)[tid];
      S.hist[0][2 * tid] = h2.x; S.hist[0][2 * tid + 1] = h2.y;
      S.hist[1][2 * tid] = 0; S.hist[1][2 * tid + 1] = 0;
      nvalid = n;   // every entry of a score segment is valid
      // the first find_bin barrier publishes both arrays
    } else {
      // ---- the leading bits every valid key shares, and the number of valid keys:
      // the radix digits start below the shared bits (scores in a narrow range, such
      // as the top candidates a merge level sees, would otherwise crowd a few bins of
      // the first digit), and a segment with no more valid keys than k keeps them
      // all. Every warp reduces the per-warp values itself after one barrier.
      uint32_t a = 0xFFFFFFFFu, o = 0u;
#pragma unroll
      for (int i = 0; i < CNT; ++i)
        if ((valid >> i) & 1u) { a &= key[i]; o |= key[i]; }
      a = __reduce_and_sync(0xffffffffu, a);
      o = __reduce_or_sync(0xffffffffu, o);
      const int c = (int)__reduce_add_sync(0xffffffffu, (uint32_t)__popc(valid));
      if (lane == 0) { S.wand[warp] = a; S.wor[warp] = o; S.wcnt[warp] = c; }
      for (int j = tid; j < 2 * kHistBins; j += kTopkThreads) (&S.hist[0][0])[j] = 0;
      __syncthreads();
      const uint32_t common = __reduce_and_sync(0xffffffffu, S.wand[lane]);
      const uint32_t any = __reduce_or_sync(0xffffffffu, S.wor[lane]);
      nvalid = (int)__reduce_add_sync(0xffffffffu, (uint32_t)S.wcnt[lane]);
      consumed = (common == any) ? 32 : __clz(common ^ any);
      pmask = consumed == 0 ? 0u : (0xFFFFFFFFu << (32 - consumed));
      prefix = common & pmask;
    }
    if (nvalid <= k) {
      // no more valid entries than k: every one of them is taken (prefix and mask 0)
      rem = count = nvalid;
      prefix = 0u; pmask = 0u;
    } else {
      rem = count = k;
      bool done = consumed == 32;   // every valid key equal: the first k by position
      // at most three digits (11 + 11 + 10 bits); the third reuses the first histogram,
      // cleared while the second digit is resolved
      for (int d = 0; d < 3 && !done; ++d) {
        const int w = min(11, 32 - consumed), sh = 32 - consumed - w;
        const uint32_t dmask = (1u << w) - 1u;
        int* h = S.hist[d & 1];
        if (!(seeded && d == 0)) {
#pragma unroll
          for (int i = 0; i < CNT; ++i)
            if (((valid >> i) & 1u) && (key[i] & pmask) == prefix) atomicAdd(&h[(key[i] >> sh) & dmask], 1);
        }
        const TopkBin b = topk_find_bin(S, h, 1 << w, rem, (d == 1 && consumed + w < 32) ? S.hist[0] : nullptr);
        rem -= b.above;
        prefix |= (uint32_t)b.bin << sh;
        pmask |= dmask << sh;
        consumed += w;
        done = b.cnt == rem || consumed == 32;
      }
    }

    // ---- ordered placement: one block scan of (above << 16 | equal) counts (each
    // total <= 16384, so no carry); an element is taken if its masked key is above the
    // prefix, or equal and among the first `rem` equal ones by position
    gt_bits = 0; eq_bits = 0;
#pragma unroll
    for (int i = 0; i < CNT; ++i) {
      const uint32_t m = key[i] & pmask;
      if (((valid >> i) & 1u) && m > prefix) gt_bits |= 1u << i;
      if (((valid >> i) & 1u) && m == prefix) eq_bits |= 1u << i;
    }
    packed = (__popc(gt_bits) << 16) | __popc(eq_bits);
    incl = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) S.wscan[warp] = incl;
    __syncthreads();
    wv = S.wscan[lane];
    wincl = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wincl, o);
      if (lane >= o) wincl += u;
    }
    if constexpr (seeded) {
      // the selection is right exactly when it takes k entries and, unless the prefix
      // covers all 32 bits, every entry equal to it under the mask
      const int total = __shfl_sync(0xffffffffu, wincl, 31);
      const int tg = total >> 16, te = total & 0xffff;
      if (!(rem >= 0 && tg + min(rem, te) == k && (rem >= te || pmask == 0xFFFFFFFFu))) return false;
    }
  }
  const int excl = __shfl_sync(0xffffffffu, wincl - wv, warp) + incl - packed;
  int rg = excl >> 16, re = excl & 0xffff;
  const bool lists = MODE == kChunks || (MODE == kMerge && L.n_out > 1);
  if (gt_bits | eq_bits) {
#pragma unroll
    for (int i = 0; i < CNT; ++i) {
      const bool is_gt = (gt_bits >> i) & 1u, is_eq = (eq_bits >> i) & 1u;
      if (is_gt || (is_eq && re < rem)) {
        const int64_t o = out_base + rg + min(re, rem);
        const int e = e0 + i;
        const int v = (MODE == kMerge) ? pos_s[e] : idx_offset + e;
        if (lists) { L.cand_idx_out[o] = v; L.cand_key_out[o] = key[i]; }
        else L.idx_out[o] = v;
      }
      if (is_gt) ++rg;
      if (is_eq) ++re;
    }
  }
  for (int j = count + tid; j < k; j += kTopkThreads) {
    if (lists) { L.cand_idx_out[out_base + j] = -1; L.cand_key_out[out_base + j] = 0u; }
    else L.idx_out[out_base + j] = -1;
  }
  return true;
}

// Runs of 4, 8 or 16 entries per thread, whichever spreads the segment over the most
// threads; a seeded selection the final counts reject is done again unseeded.
template <int MODE, int CNT, bool kSeeded>
__device__ __forceinline__ void topk_select_seeded(const TopkLaunch& L, int n, int64_t in_base, int64_t out_base,
                                                   int idx_offset, TopkShared& S, int* pos_s, const int* hrow) {
  if (topk_select<CNT, MODE, kSeeded>(L, n, in_base, out_base, idx_offset, S, pos_s, hrow)) return;
  if constexpr (kSeeded) {
    if (threadIdx.x == 0 && L.err) atomicAdd(L.err + kHistRejectedWord, 1);
    __syncthreads();   // every warp is done with the shared arrays of the first pass
    topk_select<CNT, MODE, false>(L, n, in_base, out_base, idx_offset, S, pos_s, nullptr);
  }
}
template <int MODE, bool kSeeded>
__device__ __forceinline__ void topk_select_runs(const TopkLaunch& L, int n, int64_t in_base, int64_t out_base,
                                                 int idx_offset, TopkShared& S, int* pos_s, const int* hrow) {
  if (n <= 4 * kTopkThreads) topk_select_seeded<MODE, 4, kSeeded>(L, n, in_base, out_base, idx_offset, S, pos_s, hrow);
  else if (n <= 8 * kTopkThreads) topk_select_seeded<MODE, 8, kSeeded>(L, n, in_base, out_base, idx_offset, S, pos_s, hrow);
  else topk_select_seeded<MODE, 16, kSeeded>(L, n, in_base, out_base, idx_offset, S, pos_s, hrow);
}

// kSeeded (kDirect, kChunks): L.hist holds the indexer's first-digit histograms.
template <int MODE, bool kSeeded>
__global__ void __launch_bounds__(kTopkThreads, 1) topk_kernel(const TopkLaunch L) {
  __shared__ TopkShared S;
  __shared__ int row_len_s, row_pos_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int t, c = 0, grp = 0;
  if (MODE == kChunks) { t = blockIdx.x / L.nl; c = L.c0 + blockIdx.x % L.nl; }
  else if (MODE == kMerge) { t = blockIdx.x / L.n_out; grp = blockIdx.x % L.n_out; }
  else t = blockIdx.x;

  // Row length from the geometry (an input of the call, not of the preceding
  // kernel), found by one warp while the scores may still be in flight.
  if (warp == 0) {
    const QueryInfo qi = query_info_warp(L.g, t);
    if (lane == 0) {
      int n, pos = -1;
      if (!qi.ok && MODE != kMerge) record_error(L.err, kDevBadIndex);
      if (qi.ok) pos = qi.pos;
      if (MODE == kMerge) n = min(L.fan, L.n_in - grp * L.fan) * L.k;
      else if (MODE == kChunks) n = max(0, min(L.chunk, pos + 1 - c * L.chunk));
      else n = pos + 1;
      row_len_s = n;
      row_pos_s = pos;
    }
  }
  griddep_launch_dependents();
  griddep_wait();   // scores (or candidates) come from the preceding kernel
  // The indexer's first-digit histogram of this row (or chunk), if it counted one; it
  // is zeroed for the next step once read, whatever path the row takes.
  int* hrow = kSeeded ? L.hist + ((int64_t)t * L.hist_chunks + c) * kHistBins : nullptr;
  __syncthreads();
  const int n = row_len_s;
  const int k = L.k;

  // Where the row's entries and outputs live.
  const int64_t in_base = (MODE == kDirect) ? (int64_t)t * L.score_stride
                        : (MODE == kChunks) ? (int64_t)t * L.score_stride + (int64_t)(c - L.c0) * L.chunk
                                              : ((int64_t)t * L.n_in + (int64_t)grp * L.fan) * k;
  const int64_t out_base = (MODE == kChunks) ? ((int64_t)t * L.nchunks + c) * k
                         : (MODE == kMerge && L.n_out > 1) ? ((int64_t)t * L.n_out + grp) * k
                                                             : (int64_t)t * k;
  const int idx_offset = (MODE == kChunks) ? c * L.chunk : 0;

  if (kSeeded && n <= k) reinterpret_cast<int2*>(hrow)[tid] = make_int2(0, 0);   // not read
  if (MODE == kMerge && L.n_out == 1 && row_pos_s + 1 <= k) {
    // every valid key is kept: positions 0..pos in order (no candidate is read)
    for (int i = tid; i < k; i += kTopkThreads) L.idx_out[out_base + i] = i <= row_pos_s ? i : -1;
    return;
  }
  if (n <= k) {
    // Everything valid is taken; positions are already ascending (a single merged
    // list is copied as it is: its valid entries come first).
    for (int i = tid; i < k; i += kTopkThreads) {
      if (MODE == kChunks) {
        const bool v = i < n;
        L.cand_key_out[out_base + i] = v ? orderable_key(L.scores[in_base + i]) : 0u;
        L.cand_idx_out[out_base + i] = v ? idx_offset + i : -1;
      } else if (MODE == kDirect) {
        L.idx_out[out_base + i] = i < n ? i : -1;
      } else if (L.n_out > 1) {
        L.cand_key_out[out_base + i] = L.cand_key_in[in_base + i];
        L.cand_idx_out[out_base + i] = L.cand_idx_in[in_base + i];
      } else {
        L.idx_out[out_base + i] = L.cand_idx_in[in_base + i];
      }
    }
    return;
  }
  // Dynamic shared memory (merges only): the input candidates' positions (n).
  extern __shared__ int4 dyn_s[];
  topk_select_runs<MODE, kSeeded>(L, n, in_base, out_base, idx_offset, S, reinterpret_cast<int*>(dyn_s), hrow);
  if (kSeeded) reinterpret_cast<int2*>(hrow)[tid] = make_int2(0, 0);   // each thread read its own two
}

// ------------------------------------------------------------------ host side
int topk_chunk_len() { return kTopkCapacity; }

// Lists merged per group: as many whole lists of k as one CTA holds.
// Lists merged per group: at most four (a merge CTA of 4 x 2048 candidates is much
// quicker than one of 8 x 2048, and a level more costs less than that on these rows),
// and at most what one CTA holds.
int topk_fan_in(int k) { return kTopkCapacity / k < 4 ? kTopkCapacity / k : 4; }

// Merge levels after the chunk pass for rows of up to max_seq_len (0: no chunking).
int topk_merge_levels(int max_seq_len, int k) {
  if (max_seq_len <= kTopkCapacity) return 0;
  const int fan = topk_fan_in(k);
  if (fan < 2) return -1;
  int lists = (max_seq_len + kTopkCapacity - 1) / kTopkCapacity, levels = 0;
  while (lists > 1) { lists = (lists + fan - 1) / fan; ++levels; }
  return levels;
}

// Candidate storage: the chunk pass's lists (buffer A), and the lists of the first
// merge level when a second level follows (buffer B); later levels alternate.
static size_t topk_list_bytes(int64_t T, int64_t lists, int k) {
  return (size_t)(T * lists * k) * (sizeof(uint32_t) + sizeof(int));
}

size_t topk_workspace_bytes(int T, int max_seq_len, int k) {
  const int levels = topk_merge_levels(max_seq_len, k);
  if (levels <= 0) return 0;
  const int64_t nch = (max_seq_len + kTopkCapacity - 1) / kTopkCapacity;
  size_t bytes = (topk_list_bytes(T, nch, k) + 255) / 256 * 256;
  if (levels >= 2) bytes += topk_list_bytes(T, (nch + topk_fan_in(k) - 1) / topk_fan_in(k), k);
  return bytes;
}

// Dynamic shared memory of one launch: for merges, the positions of one segment's
// input candidates.
static size_t topk_smem_bytes(int seg_len, bool merge) {
  return merge ? (size_t)seg_len * 4 : 0;
}

static cudaError_t launch_topk_kernel(const TopkLaunch& L, int grid, int seg_len, bool pdl, cudaStream_t st) {
  const size_t smem = topk_smem_bytes(seg_len < kTopkCapacity ? seg_len : kTopkCapacity, L.mode == kMerge);
  const bool seeded = L.hist != nullptr && L.mode != kMerge;
  auto kern = L.mode == kDirect ? (seeded ? topk_kernel<kDirect, true> : topk_kernel<kDirect, false>)
            : L.mode == kChunks ? (seeded ? topk_kernel<kChunks, true> : topk_kernel<kChunks, false>)
                                : topk_kernel<kMerge, false>;
  // the 48 KB default covers static and dynamic shared memory together
  if (smem + sizeof(TopkShared) + 64 > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // The attention kernel that follows needs the whole shared-memory carveout; an SM
  // left in the same configuration takes its CTAs without reconfiguring.
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
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
  return cudaLaunchKernelEx(&cfg, kern, L);
}

int topk_row_chunks(int max_seq_len) { return max_seq_len <= kTopkCapacity ? 1 : (max_seq_len + kTopkCapacity - 1) / kTopkCapacity; }

size_t topk_hist_bytes(int T, int max_seq_len) {
  return (size_t)T * topk_row_chunks(max_seq_len) * kHistBins * sizeof(int);
}

cudaError_t topk_chunks_launch(const GeomDev& g, const float* scores, int64_t stride, int k, int c0, int nl,
                               void* scratch, int* err, bool pdl, cudaStream_t st, int* hist) {
  const int nch = (g.max_seq_len + kTopkCapacity - 1) / kTopkCapacity;
  TopkLaunch L{};
  L.g = g; L.k = k; L.mode = kChunks; L.scores = scores; L.score_stride = stride; L.err = err;
  L.hist = hist; L.hist_chunks = nch;
  L.chunk = kTopkCapacity; L.c0 = c0; L.nl = nl; L.nchunks = nch;
  L.cand_key_out = reinterpret_cast<uint32_t*>(scratch);
  L.cand_idx_out = reinterpret_cast<int*>(L.cand_key_out + (size_t)g.T * nch * k);
  return launch_topk_kernel(L, g.T * nl, kTopkCapacity, pdl, st);
}

cudaError_t topk_merge_launch(const GeomDev& g, int k, int* idx, void* scratch, int* err, bool pdl, cudaStream_t st) {
  const int nch = (g.max_seq_len + kTopkCapacity - 1) / kTopkCapacity;
  const int fan = topk_fan_in(k);
  uint8_t* buf[2] = {reinterpret_cast<uint8_t*>(scratch),
                     reinterpret_cast<uint8_t*>(scratch) + (topk_list_bytes(g.T, nch, k) + 255) / 256 * 256};
  int lists = nch, src = 0;
  while (true) {
    const int out = (lists + fan - 1) / fan;
    TopkLaunch L{};
    L.g = g; L.k = k; L.mode = kMerge; L.err = err;
    L.n_in = lists; L.fan = fan; L.n_out = out;
    L.cand_key_in = reinterpret_cast<const uint32_t*>(buf[src]);
    L.cand_idx_in = reinterpret_cast<const int*>(L.cand_key_in + (size_t)g.T * lists * k);
    if (out > 1) {
      L.cand_key_out = reinterpret_cast<uint32_t*>(buf[src ^ 1]);
      L.cand_idx_out = reinterpret_cast<int*>(L.cand_key_out + (size_t)g.T * out * k);
    } else {
      L.idx_out = idx;
    }
    const cudaError_t e = launch_topk_kernel(L, g.T * out, (lists < fan ? lists : fan) * k, pdl, st);
    if (e != cudaSuccess || out == 1) return e;
    pdl = true;   // each level follows the one just launched
    lists = out;
    src ^= 1;
  }
}

cudaError_t topk_launch(const GeomDev& g, const float* scores, int64_t stride, int k, int* idx,
                        void* scratch, int* err, bool pdl, cudaStream_t st, int* hist) {
  if (g.max_seq_len <= kTopkCapacity) {
    TopkLaunch L{};
    L.g = g; L.k = k; L.mode = kDirect; L.scores = scores; L.score_stride = stride; L.idx_out = idx; L.err = err;
    L.hist = hist; L.hist_chunks = 1;
    return launch_topk_kernel(L, g.T, g.max_seq_len, pdl, st);
  }
  const int nch = (g.max_seq_len + kTopkCapacity - 1) / kTopkCapacity;
  cudaError_t e = topk_chunks_launch(g, scores, stride, k, 0, nch, scratch, err, pdl, st, hist);
  if (e != cudaSuccess) return e;
  return topk_merge_launch(g, k, idx, scratch, err, true, st);   // follows the chunk pass just launched
}

}  // namespace dsa
