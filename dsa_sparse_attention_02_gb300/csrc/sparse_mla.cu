// Sparse absorbed-MLA attention over the selected latent rows, with a split
// combine (lmdeploy "feat: support GLM-5.2", Five-layer ablations: zero-copy BF16
// sparse MLA over the paged cache, FP8 cache path; mlx-lm "GLM-5.2 (glm_moe_dsa)
// inference", small-L gather commit: k = v = latent, unembed after; lmdeploy
// "glm5.3-flash support", Operator-level gains: negative indices are padding).
//
// For query t and head h over its selected positions s_i (idx row, -1 skipped):
//   z_i = sm_scale * q[t,h,:] . kv[s_i,:]   (576 wide)
//   out[t,h,:] = sum_i softmax(z)_i kv[s_i, 0:512],  lse[t,h] = ln sum_i exp(z_i)
//
// Work: the T x C list of (query, 128-key chunk) pairs, C = ceil(k/128), split
// evenly over a persistent grid. A chunk's 128 selected rows live in shared
// memory as 128-byte-swizzled K-major atoms of 64 bf16 columns: four "pair"
// slots of two atoms (latent columns 0..511) and one RoPE atom (512..575). The
// slots form rings (5 pair slots, 2 RoPE slots), so the next chunk's RoPE atom
// and first pair load while the current chunk computes, and its other pairs
// load as soon as the current chunk's PV MMAs release theirs.
//   * a resolver warp maps each chunk's 128 logical positions to physical cache
//     rows through the block table (-1 for padding or out-of-range entries) up
//     to four chunks ahead, into a shared-memory row table that the producer
//     and the softmax warps read.
//   * bf16 cache: two producer warps copy the rows with 16-byte cp.async, slot
//     by slot (RoPE atom, then the four pairs), each warp half of every slot;
//     padding rows are zero-filled. Each producer thread ends a slot with
//     cp.async.mbarrier.arrive.noinc, so the slot's full barrier completes when
//     the copies have landed and producers never wait on their own copies; the
//     MMA thread fences the generic->async proxy after each wait. (TMA
//     tile::gather4 of 4 x 128-byte row pieces measured at half the bandwidth
//     of this on the same access pattern.)
//   * e4m3 cache: three producer warps load the 656-byte records, dequantize
//     (code * per-128 scale) to bf16 and store into the same slots.
//   * one MMA thread: S^T = KV . Q^T on tcgen05 (M = 128 keys, N = 16 heads,
//     K = 576) into TMEM, then O^T = V^T . P^T (M = 128 latent columns x 4
//     blocks, N = 16, K = 128 keys), V^T read MN-major from the pair slots.
//   * 4 softmax warps (TMEM lane = key for S) run the online softmax per head in
//     the exp2 domain and write P^T as bf16 for the second MMA. O^T accumulates
//     in TMEM across a query's chunks. The reference max moves only when a
//     chunk's max exceeds it by more than 2^8 (p <= 256 otherwise); then the
//     softmax warps rescale O in TMEM (lane = latent column) before releasing P.
//     S(i) completing implies PV(i-1) completed (a commit tracks every earlier
//     MMA of the issuing thread), so that rescale needs no further wait.
// A CTA that holds every chunk of a query writes the final bf16 output; other
// segments write (unnormalized O, running max, sum) partials that the combine
// kernel merges with log-sum-exp weights.
#include <cstdint>
#include <cuda_bf16.h>
#include "kernels.cuh"

namespace dsa {

constexpr int kMlaHeads = 16;                       // heads per CTA (MMA N)
constexpr int kMlaKeys = 128;                       // keys per chunk (MMA M)
constexpr int kAtomBytes = kMlaKeys * 128;          // 16 KB: 128 rows x 64 bf16
constexpr int kPairBytes = 2 * kAtomBytes;          // 32 KB
constexpr int kPairSlots = 5;
constexpr int kRopeSlots = 2;
constexpr int kQAtomBytes = kMlaHeads * 128;        // 2 KB
constexpr int kQBufBytes = 9 * kQAtomBytes;         // 18 KB
constexpr int kPBufBytes = 2 * kQAtomBytes;         // P^T: 16 heads x 128 keys bf16 = 4 KB
constexpr int kMlaSmemBytes =
    1024 + kPairSlots * kPairBytes + kRopeSlots * kAtomBytes + kQBufBytes + 2 * kPBufBytes;
// Twelve warps, 168 registers each (three per SM sub-partition):
//   warps 0-3   softmax (one per TMEM lane quarter)
//   warps 4-7   producers (one per sub-partition, so that copy issue runs on all four)
//   warp  8     MMA issuer; warp 9 row resolver; warps 10-11 idle
constexpr int kMlaThreads = 384;
constexpr int kProdWarp0 = 4;
constexpr int kProdWarps = 4;
constexpr int kMmaWarp = 8;
constexpr int kResolverWarp = 9;
constexpr int kRowBufs = 4;                         // row-table ring depth (chunks)
constexpr int kMlaTmemCols = 128;                   // S: 2 x 16, O: 64
constexpr float kRescaleLog2 = 8.f;                 // lazy rescale threshold (log2 units)
constexpr float kLn2 = 0.6931471805599453f;

// Bounded group barrier over the 4 softmax warps (one arrive per warp).
struct GroupSync {
  uint32_t bar;
  uint32_t phase;
  __device__ __forceinline__ bool sync(volatile int* abort, int* err) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase, abort, err);
    phase ^= 1;
    __syncwarp();
    return ok;
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// e4m3 code -> fp32, exact (sign, 4-bit exponent with bias 7, 3-bit mantissa;
// exponent 0 encodes subnormals m * 2^-9; S.1111.111 is NaN).
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const uint32_t sign = (c & 0x80u) << 24;
  const uint32_t em = c & 0x7Fu;
  float v;
  if (em == 0x7Fu) v = __uint_as_float(0x7FC00000u);
  else if ((em >> 3) == 0) v = (float)(em & 7u) * 0.001953125f;            // m * 2^-9
  else v = __uint_as_float((((em >> 3) + 120u) << 23) | ((em & 7u) << 20));  // rebias 7 -> 127
  return __uint_as_float(__float_as_uint(v) | sign);
}

// 2^x with the MUFU ex2 instruction (inputs here are <= 8 or -inf).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Max over the 32 lanes of 16 values at once (a transposing butterfly: 16 shuffles
// instead of 80). On return, lanes h and h+16 hold the max of value h.
__device__ __forceinline__ float warp_max16(const float (&v)[16]) {
  const int lane = threadIdx.x & 31;
  float a[8];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float send = up ? v[k] : v[k + 8];
      const float keep = up ? v[k + 8] : v[k];
      a[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
  }
  float b[4];
  {
    const bool up = lane & 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float send = up ? a[k] : a[k + 4];
      const float keep = up ? a[k + 4] : a[k];
      b[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
  }
  float c[2];
  {
    const bool up = lane & 4;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float send = up ? b[k] : b[k + 2];
      const float keep = up ? b[k + 2] : b[k];
      c[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
  }
  float d;
  {
    const bool up = lane & 2;
    const float send = up ? c[0] : c[1];
    const float keep = up ? c[1] : c[0];
    d = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  }
  return fmaxf(d, __shfl_xor_sync(0xffffffffu, d, 1));
}

struct ChunkPos {
  int64_t chunk;
  int t, cq;
  bool first, last;
};

// Physical cache row of the selected position at offset e of query t's index row,
// or -1 for padding / out-of-range entries (reported).
__device__ __forceinline__ int64_t selected_row(const MlaArgs& A, const QueryInfo& qi, int t, int e) {
  if (!qi.ok || e >= A.k) return -1;
  const int s = __ldg(A.idx + (int64_t)t * A.k + e);
  if (s < 0) return -1;
  const int64_t row = s < qi.len ? physical_row(A.g, qi.b, s) : -1;
  if (row < 0) record_error(A.err, kDevBadIndex);
  return row;
}

template <bool kFp8Kv>
__global__ void __launch_bounds__(kMlaThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap map_q, const MlaArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* pair_buf = smem;                                         // 5 x 32 KB
  uint8_t* rope_buf = pair_buf + kPairSlots * kPairBytes;           // 2 x 16 KB
  uint8_t* q_buf = rope_buf + kRopeSlots * kAtomBytes;              // 18 KB
  uint8_t* p_buf = q_buf + kQBufBytes;                              // 2 x 4 KB

  __shared__ uint64_t pair_full[kPairSlots], pair_empty[kPairSlots], rope_full[kRopeSlots], rope_empty[kRopeSlots];
  __shared__ uint64_t q_full, q_empty;
  __shared__ uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2], o_full, o_free, grp_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  __shared__ __align__(16) float red[2][4][kMlaHeads];
  __shared__ __align__(16) int rows_s[kRowBufs][kMlaKeys];   // physical row per key of a chunk, -1 = none
  __shared__ uint64_t rows_full[kRowBufs], rows_empty[kRowBufs];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GeomDev& g = A.g;
  const int G = gridDim.x;
  const int hg = blockIdx.y;
  const int h_eff = min(kMlaHeads, A.H - hg * kMlaHeads);
  const int64_t c_begin = split_begin(blockIdx.x, A.n_chunks, G);
  const int64_t c_end = split_begin(blockIdx.x + 1, A.n_chunks, G);
  const int n_mine = (int)(c_end - c_begin);
  const int slot_producers = 32 * kProdWarps;   // one arrival per producer thread per slot fill

  auto chunk_pos = [&](int i) {
    ChunkPos cp;
    cp.chunk = c_begin + i;
    cp.t = (int)(cp.chunk / A.C);
    cp.cq = (int)(cp.chunk - (int64_t)cp.t * A.C);
    cp.first = (i == 0) || (cp.cq == 0);
    cp.last = (i == n_mine - 1) || (cp.cq == A.C - 1);
    return cp;
  };

  if (tid == 0) {
    abort_flag = 0;
    for (int j = 0; j < kPairSlots; ++j) { mbar_init(smem_u32(&pair_full[j]), slot_producers); mbar_init(smem_u32(&pair_empty[j]), 1); }
    for (int j = 0; j < kRopeSlots; ++j) { mbar_init(smem_u32(&rope_full[j]), slot_producers); mbar_init(smem_u32(&rope_empty[j]), 1); }
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&q_empty), 1);
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_u32(&s_full[j]), 1);
      mbar_init(smem_u32(&s_empty[j]), 4);
      mbar_init(smem_u32(&p_full[j]), 4);
      mbar_init(smem_u32(&p_empty[j]), 1);
    }
    mbar_init(smem_u32(&o_full), 1);     // one phase per chunk's PV
    mbar_init(smem_u32(&o_free), 4);     // softmax warps have read O at a segment end
    mbar_init(smem_u32(&grp_bar), 4);
    for (int j = 0; j < kRowBufs; ++j) {
      // written by the resolver warp, read by the producer and softmax warps
      mbar_init(smem_u32(&rows_full[j]), 1);
      mbar_init(smem_u32(&rows_empty[j]), 4 + kProdWarps);
    }
    fence_mbar_init();
  }
  // Query rows >= h_eff stay zero (TMA writes h_eff rows per atom).
  for (int i = tid; i < kQBufBytes / 16; i += kMlaThreads) reinterpret_cast<int4*>(q_buf)[i] = make_int4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == kMmaWarp) { tmem_alloc(smem_u32(&tmem_base_s), kMlaTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tmem_s = tmem;          // + 16 * buf
  const uint32_t tmem_o = tmem + 32;     // + 16 * mb

  if (warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps) {
    // ================================================================ producers
    // Warp pw copies rows [32*pw, 32*pw+32) of every slot. bf16: 16-byte cp.async
    // (zero-fill for padding), slot completion through cp.async.mbarrier.arrive.noinc.
    // e4m3: the RoPE atom by cp.async as well; the latent pairs are loaded,
    // dequantized to bf16 and stored, then each thread arrives.
    const int pw = warp - kProdWarp0;
    int seg = 0;
    auto slot_acquire = [&](uint32_t bar, uint32_t parity) -> bool {   // warp-uniform bounded wait
      int ok = 1;
      if (lane == 0) ok = mbar_wait(bar, parity, &abort_flag, A.err) ? 1 : 0;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    const size_t row_bytes = kFp8Kv ? (size_t)kFp8Record : (size_t)(kDimQK * 2);
    const size_t rope_off = kFp8Kv ? (size_t)(kDimLatent + 16) : (size_t)(kDimLatent * 2);
    for (int i = 0; i < n_mine; ++i) {
      const ChunkPos cp = chunk_pos(i);
      if (cp.first) {
        if (pw == 0) {
          if (!slot_acquire(smem_u32(&q_empty), (seg & 1) ^ 1)) break;
          if (lane == 0) {
            const uint32_t bar = smem_u32(&q_full);
            mbar_arrive_expect_tx(bar, 9 * h_eff * 128);
            for (int a = 0; a < 9; ++a)
              tma_load_2d(smem_u32(q_buf + a * kQAtomBytes), &map_q, bar, a * 64, cp.t * A.H + hg * kMlaHeads);
          }
        }
        ++seg;
      }
      const int rb = i % kRowBufs, rs = i % kRopeSlots;
      if (!slot_acquire(smem_u32(&rows_full[rb]), (i / kRowBufs) & 1)) break;
      mbar_try_wait(smem_u32(&rows_full[rb]), (i / kRowBufs) & 1);   // acquire in every lane (phase is complete)
      const int* rows = rows_s[rb];
      const uint8_t* kv = A.kv;
      // RoPE atom: 8 lanes per row (128 B), 4 rows per instruction
      if (!slot_acquire(smem_u32(&rope_empty[rs]), ((i / kRopeSlots) & 1) ^ 1)) break;
      {
        const uint32_t dst0 = smem_u32(rope_buf + rs * kAtomBytes);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int ri = 32 * pw + 4 * j + (lane >> 3);
          const int row = rows[ri];
          const int cb = (lane & 7) * 16;
          cp_async_16(dst0 + sw128_offset(ri, cb, 0), kv + (int64_t)(row >= 0 ? row : 0) * row_bytes + rope_off + cb,
                      row >= 0 ? 16u : 0u);
        }
        cp_async_arrive_noinc(smem_u32(&rope_full[rs]));
      }
      bool stop = false;
      for (int j = 0; j < 4; ++j) {
        const int gidx = 4 * i + j, ps = gidx % kPairSlots;
        if (!slot_acquire(smem_u32(&pair_empty[ps]), ((gidx / kPairSlots) & 1) ^ 1)) { stop = true; break; }
        uint8_t* slot = pair_buf + ps * kPairBytes;
        if (!kFp8Kv) {
          // 16 lanes per row (256 B of the pair), 2 rows per instruction
          const uint32_t dst0 = smem_u32(slot);
#pragma unroll 4
          for (int jj = 0; jj < 16; ++jj) {
            const int ri = 32 * pw + 2 * jj + (lane >> 4);
            const int row = rows[ri];
            const int cb = (lane & 15) * 16;
            cp_async_16(dst0 + sw128_offset(ri, cb, kAtomBytes), kv + (int64_t)(row >= 0 ? row : 0) * row_bytes + j * 256 + cb,
                        row >= 0 ? 16u : 0u);
          }
          cp_async_arrive_noinc(smem_u32(&pair_full[ps]));
        } else {
          // 8 lanes per row: lane part p dequantizes codes 16p..16p+15 of the pair's 128
          const int part = lane & 7, sub = lane >> 3;
          uint4 c[8];
          float sc[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int row = rows[32 * pw + 4 * jj + sub];
            c[jj] = make_uint4(0, 0, 0, 0);
            sc[jj] = 0.f;
            if (row >= 0) {
              const uint8_t* rec = kv + (int64_t)row * kFp8Record;
              c[jj] = __ldg(reinterpret_cast<const uint4*>(rec + 128 * j) + part);
              sc[jj] = __ldg(reinterpret_cast<const float*>(rec + kDimLatent) + j);
            }
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int key = 32 * pw + 4 * jj + sub;
            const uint32_t w4[4] = {c[jj].x, c[jj].y, c[jj].z, c[jj].w};
            uint32_t pk[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t wv = w4[q];
              pk[2 * q] = pack_bf16x2(e4m3_to_f32(wv & 0xFF) * sc[jj], e4m3_to_f32((wv >> 8) & 0xFF) * sc[jj]);
              pk[2 * q + 1] = pack_bf16x2(e4m3_to_f32((wv >> 16) & 0xFF) * sc[jj], e4m3_to_f32(wv >> 24) * sc[jj]);
            }
            // pair column 16*part .. 16*part+15 -> atom part/4, bytes 32*(part%4) .. +31
            const int col_byte = (part >> 2) * 128 + (part & 3) * 32;
            *reinterpret_cast<uint4*>(slot + sw128_offset(key, col_byte, kAtomBytes)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(slot + sw128_offset(key, col_byte + 16, kAtomBytes)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&pair_full[ps]));
        }
      }
      if (stop) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&rows_empty[rb]));
    }
  } else if (warp == kResolverWarp) {
    // ================================================================ row resolver
    int t_cached = -1;
    QueryInfo qi{};
    for (int i = 0; i < n_mine; ++i) {
      const ChunkPos cp = chunk_pos(i);
      if (cp.t != t_cached) { qi = query_info_warp(g, cp.t); t_cached = cp.t; }
      const int rb = i % kRowBufs;
      int rr[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) rr[m] = (int)selected_row(A, qi, cp.t, cp.cq * kMlaKeys + 4 * lane + m);
      if (!mbar_wait(smem_u32(&rows_empty[rb]), ((i / kRowBufs) & 1) ^ 1, &abort_flag, A.err)) break;
      *reinterpret_cast<int4*>(&rows_s[rb][4 * lane]) = make_int4(rr[0], rr[1], rr[2], rr[3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&rows_full[rb]));
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc(128, kMlaHeads, kFmtBF16, kFmtBF16, 0, 0);
      constexpr uint32_t idesc_o = make_idesc(128, kMlaHeads, kFmtBF16, kFmtBF16, 1, 0);
      const uint32_t pair0 = smem_u32(pair_buf), rope0 = smem_u32(rope_buf), q0 = smem_u32(q_buf);
      int seg = -1;
      for (int i = 0; i < n_mine; ++i) {
        const ChunkPos cp = chunk_pos(i);
        if (cp.first) ++seg;
        const int sb = i & 1, rs = i % kRopeSlots;
        const uint32_t ph2 = (i >> 1) & 1;
        if (!mbar_wait(smem_u32(&s_empty[sb]), ph2 ^ 1, &abort_flag, A.err)) break;
        if (cp.first && !mbar_wait(smem_u32(&q_full), seg & 1, &abort_flag, A.err)) break;
        if (!mbar_wait(smem_u32(&rope_full[rs]), (i / kRopeSlots) & 1, &abort_flag, A.err)) break;
        fence_proxy_async_smem();   // slot filled through the generic proxy (cp.async / st.shared)
        tc_fence_after();
        const uint32_t d_s = tmem_s + sb * 16;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16_ss(d_s, smem_desc(rope0 + rs * kAtomBytes + kk * 32, 0, 1024, kSwizzle128B),
                     smem_desc(q0 + 8 * kQAtomBytes + kk * 32, 0, 1024, kSwizzle128B), idesc_s, kk != 0);
        mma_commit(smem_u32(&rope_empty[rs]));
        bool stop = false;
        for (int j = 0; j < 4; ++j) {
          const int gidx = 4 * i + j, ps = gidx % kPairSlots;
          if (!mbar_wait(smem_u32(&pair_full[ps]), (gidx / kPairSlots) & 1, &abort_flag, A.err)) { stop = true; break; }
          fence_proxy_async_smem();
          tc_fence_after();
#pragma unroll
          for (int a2 = 0; a2 < 2; ++a2) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ss(d_s, smem_desc(pair0 + ps * kPairBytes + a2 * kAtomBytes + kk * 32, 0, 1024, kSwizzle128B),
                         smem_desc(q0 + (2 * j + a2) * kQAtomBytes + kk * 32, 0, 1024, kSwizzle128B), idesc_s, 1);
          }
        }
        if (stop) break;
        mma_commit(smem_u32(&s_full[sb]));
        if (cp.last) mma_commit(smem_u32(&q_empty));
        if (!mbar_wait(smem_u32(&p_full[sb]), ph2, &abort_flag, A.err)) break;
        // a new segment's first PV overwrites O: the previous segment's O must have been read
        if (cp.first && seg > 0 && !mbar_wait(smem_u32(&o_free), (seg - 1) & 1, &abort_flag, A.err)) break;
        tc_fence_after();
        const uint32_t p0 = smem_u32(p_buf + sb * kPBufBytes);
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
          const int ps = (4 * i + mb) % kPairSlots;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t ad = smem_desc(pair0 + ps * kPairBytes + ks * 2048, kAtomBytes, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(p0 + (ks >> 2) * kQAtomBytes + (ks & 3) * 32, 0, 1024, kSwizzle128B);
            mma_f16_ss(tmem_o + mb * 16, ad, bd, idesc_o, (ks != 0 || !cp.first) ? 1u : 0u);
          }
          mma_commit(smem_u32(&pair_empty[ps]));
        }
        mma_commit(smem_u32(&o_full));
        mma_commit(smem_u32(&p_empty[sb]));
      }
    }
  } else if (warp < 4) {
    // ================================================================ softmax warps 0-3
    GroupSync gs{smem_u32(&grp_bar), 0};
    int red_i = 0;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float neg_inf = -__int_as_float(0x7f800000);
    float m[kMlaHeads], l[kMlaHeads];
    for (int i = 0; i < n_mine; ++i) {
      const ChunkPos cp = chunk_pos(i);
      const int sb = i & 1;
      const uint32_t ph2 = (i >> 1) & 1;
      if (cp.first) {
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) { m[h] = neg_inf; l[h] = 0.f; }
      }
      // validity of this thread's key from the row table
      const int rb = i % kRowBufs;
      if (!mbar_wait(smem_u32(&rows_full[rb]), (i / kRowBufs) & 1, &abort_flag, A.err)) break;
      const bool valid = rows_s[rb][tid] >= 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&rows_empty[rb]));
      if (!mbar_wait(smem_u32(&s_full[sb]), ph2, &abort_flag, A.err)) break;
      tc_fence_after();
      float z[kMlaHeads];
      tmem_ld16(tmem_s + sb * 16 + lane_off, z);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_empty[sb]));
      // chunk max per head across the 128 keys
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h) z[h] = valid ? z[h] * A.scale_log2 : neg_inf;
      {
        // after the butterfly, lanes 2h' and 2h'+1 hold the warp max of head hidx below
        // (exchange distances 16, 8, 4, 2 select head bits 3, 2, 1, 0)
        const float wm = warp_max16(z);
        const int hidx = ((lane >> 4) & 1) << 3 | ((lane >> 3) & 1) << 2 | ((lane >> 2) & 1) << 1 | ((lane >> 1) & 1);
        if ((lane & 1) == 0) red[red_i][warp][hidx] = wm;
      }
      if (!gs.sync(&abort_flag, A.err)) break;
      // move the reference max only where this chunk exceeds it by more than 2^8
      float alpha[kMlaHeads];
      bool any_raise = false;
      {
        float cmv[kMlaHeads];
#pragma unroll
        for (int q4 = 0; q4 < kMlaHeads / 4; ++q4) {
          const float4 r0 = *reinterpret_cast<const float4*>(&red[red_i][0][4 * q4]);
          const float4 r1 = *reinterpret_cast<const float4*>(&red[red_i][1][4 * q4]);
          const float4 r2 = *reinterpret_cast<const float4*>(&red[red_i][2][4 * q4]);
          const float4 r3 = *reinterpret_cast<const float4*>(&red[red_i][3][4 * q4]);
          cmv[4 * q4 + 0] = fmaxf(fmaxf(r0.x, r1.x), fmaxf(r2.x, r3.x));
          cmv[4 * q4 + 1] = fmaxf(fmaxf(r0.y, r1.y), fmaxf(r2.y, r3.y));
          cmv[4 * q4 + 2] = fmaxf(fmaxf(r0.z, r1.z), fmaxf(r2.z, r3.z));
          cmv[4 * q4 + 3] = fmaxf(fmaxf(r0.w, r1.w), fmaxf(r2.w, r3.w));
        }
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) {
          const float cm = cmv[h];
          alpha[h] = 1.f;
          if (cm > m[h] + kRescaleLog2) {       // also true for the first finite max (m = -inf)
            alpha[h] = (m[h] == neg_inf) ? 0.f : fast_exp2(m[h] - cm);
            any_raise = true;
            m[h] = cm;
          }
          l[h] *= alpha[h];
          z[h] = (z[h] == neg_inf) ? 0.f : fast_exp2(z[h] - m[h]);   // z now holds p <= 256
          l[h] += z[h];
        }
      }
      red_i ^= 1;
      if (any_raise && !cp.first) {
        // O in TMEM holds this segment's earlier chunks (their PVs are complete: S(i)
        // was committed after them); scale the raised heads' columns by alpha.
#pragma unroll
        for (int mb = 0; mb < 4; ++mb) {
          float ov[16];
          tmem_ld16(tmem_o + mb * 16 + lane_off, ov);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < kMlaHeads; ++h) ov[h] *= alpha[h];
          tmem_st16(tmem_o + mb * 16 + lane_off, ov);
        }
        tmem_st_wait();
      }
      // P^T (K-major: row = head, 128 keys = 2 atoms) for the second MMA
      if (!mbar_wait(smem_u32(&p_empty[sb]), ph2 ^ 1, &abort_flag, A.err)) break;
      uint8_t* pb = p_buf + sb * kPBufBytes;
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h)
        *reinterpret_cast<__nv_bfloat16*>(pb + sw128_offset(h, tid * 2, kQAtomBytes)) = __float2bfloat16_rn(z[h]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full[sb]));

      if (cp.last) {
        // total sum per head over the 128 key lanes
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) {
          const float ws = warp_sum(l[h]);
          if (lane == 0) red[red_i][warp][h] = ws;
        }
        if (!gs.sync(&abort_flag, A.err)) break;
        float lt[kMlaHeads];
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h)
          lt[h] = red[red_i][0][h] + red[red_i][1][h] + red[red_i][2][h] + red[red_i][3][h];
        red_i ^= 1;
        // O^T after this chunk's PV (lane = latent column within a 128-block),
        // streamed out one 16-column block of TMEM at a time
        if (!mbar_wait(smem_u32(&o_full), i & 1, &abort_flag, A.err)) break;
        tc_fence_after();
        const int64_t c_first = split_owner((int64_t)cp.t * A.C, A.n_chunks, G);
        const int64_t c_last = split_owner((int64_t)cp.t * A.C + A.C - 1, A.n_chunks, G);
        const bool whole = c_first == c_last;
        const int hbase = hg * kMlaHeads;
        const int64_t row0 = whole ? (int64_t)cp.t * A.H + hbase : ((int64_t)cp.t + blockIdx.x) * A.H + hbase;
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) lt[h] = lt[h] > 0.f ? 1.f / lt[h] : 0.f;   // now 1/l
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
          float ov[16];
          tmem_ld16(tmem_o + mb * 16 + lane_off, ov);
          tmem_ld_wait();
          if (whole) {
            __nv_bfloat16* op = A.out + row0 * kDimLatent + mb * 128 + tid;
#pragma unroll
            for (int h = 0; h < kMlaHeads; ++h)
              if (h < h_eff) op[(int64_t)h * kDimLatent] = __float2bfloat16_rn(ov[h] * lt[h]);
          } else {
            float* op = A.o_part + row0 * kDimLatent + mb * 128 + tid;
#pragma unroll
            for (int h = 0; h < kMlaHeads; ++h)
              if (h < h_eff) op[(int64_t)h * kDimLatent] = ov[h];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&o_free));
        if (tid < h_eff) {
          float mh = m[0], inv = lt[0];
#pragma unroll
          for (int h = 1; h < kMlaHeads; ++h)
            if (tid == h) { mh = m[h]; inv = lt[h]; }
          if (whole) {
            if (A.lse) A.lse[row0 + tid] = inv > 0.f ? (mh - log2f(inv)) * kLn2 : neg_inf;
          } else {
            A.ml_part[2 * (row0 + tid)] = mh;
            A.ml_part[2 * (row0 + tid) + 1] = inv > 0.f ? 1.f / inv : 0.f;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kMlaTmemCols);
  }
}

// Merge the partial segments of every query that more than one CTA worked on.
__global__ void __launch_bounds__(128) mla_combine_kernel(const MlaArgs A, int G) {
  const int t = blockIdx.x;
  const int h = blockIdx.y;
  const int64_t c_first = split_owner((int64_t)t * A.C, A.n_chunks, G);
  const int64_t c_last = split_owner((int64_t)t * A.C + A.C - 1, A.n_chunks, G);
  if (c_first == c_last) return;
  const float neg_inf = -__int_as_float(0x7f800000);
  float mx = neg_inf;
  for (int64_t c = c_first; c <= c_last; ++c) mx = fmaxf(mx, A.ml_part[2 * ((t + c) * A.H + h)]);
  float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int64_t c = c_first; c <= c_last; ++c) {
    const int64_t r = (t + c) * A.H + h;
    const float mj = A.ml_part[2 * r], lj = A.ml_part[2 * r + 1];
    const float wgt = (mj == neg_inf) ? 0.f : exp2f(mj - mx);
    L += wgt * lj;
    const float* orow = A.o_part + r * kDimLatent;
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = fmaf(wgt, orow[j * 128 + threadIdx.x], acc[j]);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* orow = A.out + ((int64_t)t * A.H + h) * kDimLatent;
#pragma unroll
  for (int j = 0; j < 4; ++j) orow[j * 128 + threadIdx.x] = __float2bfloat16_rn(acc[j] * inv);
  if (A.lse && threadIdx.x == 0) A.lse[(int64_t)t * A.H + h] = L > 0.f ? (mx + log2f(L)) * kLn2 : neg_inf;
}

// ------------------------------------------------------------------ host side
int mla_grid(int64_t n_chunks, int num_sms) {
  return (int)(n_chunks < num_sms ? n_chunks : num_sms);
}

size_t mla_partial_bytes(int T, int H, int grid) {
  const size_t rows = (size_t)(T + grid) * H;
  return rows * kDimLatent * sizeof(float) + rows * 2 * sizeof(float);
}

cudaError_t mla_launch(bool fp8_kv, const CUtensorMap& map_q, MlaArgs A, int grid, cudaStream_t st) {
  const int hgroups = (A.H + kMlaHeads - 1) / kMlaHeads;
  auto kern = fp8_kv ? sparse_mla_kernel<true> : sparse_mla_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMlaSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<dim3(grid, hgroups), kMlaThreads, kMlaSmemBytes, st>>>(map_q, A);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (A.C > 1) {  // a query with several chunks may span CTAs
    mla_combine_kernel<<<dim3(A.g.T, A.H), 128, 0, st>>>(A, grid);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace dsa
