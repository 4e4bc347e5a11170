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
// evenly over a persistent grid. Per chunk:
//   * 3 producer warps resolve logical positions through the block table and
//     gather the 128 selected rows straight from the paged cache into one
//     128-byte-swizzled K-major tile (9 column atoms of 64 bf16): cp.async for
//     bf16 rows; for e4m3 rows a load, dequantize (code * per-128 scale) and
//     store of bf16. Padding rows are zero-filled.
//   * one MMA thread computes S^T = KV . Q^T on tcgen05 (M = 128 keys, N = 16
//     heads, K = 576) into TMEM, then, once P is ready, O^T = V^T . P^T (M = 128
//     latent columns x 4 blocks, N = 16, K = 128 keys) reading V^T MN-major
//     from the same smem tile.
//   * 4 softmax warps (TMEM lane = key) run the online softmax per head in the
//     exp2 domain, write P^T as bf16 into smem for the second MMA, and add the
//     chunk's O^T (TMEM lane = latent column) into fp32 registers after
//     rescaling.
// A CTA that holds every chunk of a query writes the final bf16 output; other
// segments write (unnormalized O, running max, sum) partials that the combine
// kernel merges with log-sum-exp weights.
#include <cstdint>
#include <cuda_bf16.h>
#include "kernels.cuh"

namespace dsa {

constexpr int kMlaHeads = 16;                       // heads per CTA (MMA N)
constexpr int kMlaKeys = 128;                       // keys per chunk (MMA M)
constexpr int kKvAtomBytes = kMlaKeys * 128;        // 16 KB: 128 rows x 64 bf16
constexpr int kKvTileBytes = 9 * kKvAtomBytes;      // 144 KB
constexpr int kQAtomBytes = kMlaHeads * 128;        // 2 KB
constexpr int kQBufBytes = 9 * kQAtomBytes;         // 18 KB
constexpr int kPBufBytes = 2 * kQAtomBytes;         // P^T: 16 heads x 128 keys bf16 = 4 KB
constexpr int kMlaSmemBytes = 1024 + kKvTileBytes + 2 * kQBufBytes + 2 * kPBufBytes;
// 8 warps: 0-3 softmax (one per TMEM lane quarter), 4-6 producers, 7 MMA. Eight
// warps put two on each SM sub-partition, which leaves room for ~200 registers.
constexpr int kMlaThreads = 256;
constexpr int kProdWarps = 3;
constexpr int kMmaWarp = 7;
constexpr int kMlaTmemCols = 256;                   // S: 2 x 16, O: 2 x 64
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

struct ChunkPos {
  int64_t chunk;
  int t, cq;
  bool first, last;
};

template <bool kFp8Kv>
__global__ void __launch_bounds__(kMlaThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap map_q, const MlaArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv_tile = smem;
  uint8_t* q_buf = smem + kKvTileBytes;                 // 2 x 18 KB
  uint8_t* p_buf = q_buf + 2 * kQBufBytes;              // 2 x 4 KB

  __shared__ uint64_t kv_full, kv_empty, q_full[2], q_empty[2];
  __shared__ uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2], o_full[2], o_empty[2], grp_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  __shared__ float red[2][4][kMlaHeads];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GeomDev& g = A.g;
  const int G = gridDim.x;
  const int hg = blockIdx.y;
  const int h_eff = min(kMlaHeads, A.H - hg * kMlaHeads);
  const int64_t c_begin = split_begin(blockIdx.x, A.n_chunks, G);
  const int64_t c_end = split_begin(blockIdx.x + 1, A.n_chunks, G);
  const int n_mine = (int)(c_end - c_begin);

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
    mbar_init(smem_u32(&kv_full), kProdWarps * 32);
    mbar_init(smem_u32(&kv_empty), 1);
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_u32(&q_full[j]), 1);
      mbar_init(smem_u32(&q_empty[j]), 1);
      mbar_init(smem_u32(&s_full[j]), 1);
      mbar_init(smem_u32(&s_empty[j]), 4);
      mbar_init(smem_u32(&p_full[j]), 4);
      mbar_init(smem_u32(&p_empty[j]), 1);
      mbar_init(smem_u32(&o_full[j]), 1);
      mbar_init(smem_u32(&o_empty[j]), 4);
    }
    mbar_init(smem_u32(&grp_bar), 4);
    fence_mbar_init();
  }
  // Query rows >= h_eff stay zero (TMA writes h_eff rows per atom).
  for (int i = tid; i < 2 * kQBufBytes / 16; i += kMlaThreads)
    reinterpret_cast<int4*>(q_buf)[i] = make_int4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == kMmaWarp) { tmem_alloc(smem_u32(&tmem_base_s), kMlaTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tmem_s = tmem;          // + 16 * buf
  const uint32_t tmem_o = tmem + 32;     // + 64 * buf, + 16 * mb

  if (warp >= 4 && warp < 4 + kProdWarps) {
    // ================================================================ producers
    // Warp pw gathers rows [r0, r1) of the chunk (43, 43, 42 rows); lane l resolves
    // rows r0 + l and r0 + 32 + l.
    const int pw = warp - 4;
    const int r0 = pw * 43, r1 = min(kMlaKeys, r0 + 43), nrows = r1 - r0;
    int seg = 0;
    for (int i = 0; i < n_mine; ++i) {
      const ChunkPos cp = chunk_pos(i);
      if (cp.first) {
        const int qb = seg & 1;
        if (pw == 0 && lane == 0) {
          if (!mbar_wait(smem_u32(&q_empty[qb]), ((seg >> 1) & 1) ^ 1, &abort_flag, A.err)) break;
          const uint32_t bar = smem_u32(&q_full[qb]);
          mbar_arrive_expect_tx(bar, 9 * h_eff * 128);
          for (int a = 0; a < 9; ++a)
            tma_load_2d(smem_u32(q_buf + qb * kQBufBytes + a * kQAtomBytes), &map_q, bar, a * 64,
                        cp.t * A.H + hg * kMlaHeads);
        }
        ++seg;
      }
      // resolve this lane's two key rows
      const QueryInfo qi = query_info(g, cp.t);
      int64_t rowv[2] = {-1, -1};
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int r = r0 + h2 * 32 + lane;
        const int e = cp.cq * kMlaKeys + r;
        if (r < r1 && qi.ok && e < A.k) {
          const int s = __ldg(A.idx + (int64_t)cp.t * A.k + e);
          if (s >= 0) {
            if (s < qi.len) rowv[h2] = physical_row(g, qi.b, s);
            if (rowv[h2] < 0) record_error(A.err, kDevBadIndex);
          }
        }
      }
      if (!mbar_wait(smem_u32(&kv_empty), (i & 1) ^ 1, &abort_flag, A.err)) break;
      if (!kFp8Kv) {
        const uint8_t* base = A.kv;
        for (int j = 0; j < nrows; ++j) {
          const int key = r0 + j;
          const int64_t pr = __shfl_sync(0xffffffffu, j < 32 ? rowv[0] : rowv[1], j & 31);
          const uint8_t* src = base + (pr >= 0 ? pr : 0) * (int64_t)(kDimQK * 2);
          const uint32_t nbytes = pr >= 0 ? 16u : 0u;
#pragma unroll
          for (int part = 0; part < 3; ++part) {
            const int c16 = part * 32 + lane;       // 16-byte chunk of the 1152-byte row
            if (c16 < 72)
              cp_async_16(smem_u32(kv_tile + sw128_offset(key, c16 * 16, kKvAtomBytes)), src + c16 * 16, nbytes);
          }
        }
        cp_async_commit();
        cp_async_wait<0>();
      } else {
        // e4m3 record: 512 latent codes | 4 fp32 scales | 64 bf16 RoPE values
        constexpr int kBatch = 8;
        for (int j0 = 0; j0 < nrows; j0 += kBatch) {
          uint4 lat[kBatch];
          float sc[kBatch];
          uint4 rope[kBatch];
#pragma unroll
          for (int jj = 0; jj < kBatch; ++jj) {
            const int j = j0 + jj;
            const int64_t pr = __shfl_sync(0xffffffffu, j < 32 ? rowv[0] : rowv[1], j & 31);
            lat[jj] = make_uint4(0, 0, 0, 0); sc[jj] = 0.f; rope[jj] = make_uint4(0, 0, 0, 0);
            if (j < nrows && pr >= 0) {
              const uint8_t* rec = A.kv + pr * (int64_t)kFp8Record;
              lat[jj] = __ldg(reinterpret_cast<const uint4*>(rec) + lane);
              sc[jj] = __ldg(reinterpret_cast<const float*>(rec + kDimLatent) + (lane >> 3));
              if (lane < 8) rope[jj] = __ldg(reinterpret_cast<const uint4*>(rec + kDimLatent + 16) + lane);
            }
          }
#pragma unroll
          for (int jj = 0; jj < kBatch; ++jj) {
            if (j0 + jj >= nrows) break;
            const int key = r0 + j0 + jj;
            const uint32_t w4[4] = {lat[jj].x, lat[jj].y, lat[jj].z, lat[jj].w};
            uint32_t packed[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t wv = w4[q];
              packed[2 * q] = pack_bf16x2(e4m3_to_f32(wv & 0xFF) * sc[jj], e4m3_to_f32((wv >> 8) & 0xFF) * sc[jj]);
              packed[2 * q + 1] = pack_bf16x2(e4m3_to_f32((wv >> 16) & 0xFF) * sc[jj], e4m3_to_f32(wv >> 24) * sc[jj]);
            }
            // latent elements 16*lane .. 16*lane+15 = bytes 32*lane .. +31 of the bf16 row
            uint8_t* d0 = kv_tile + sw128_offset(key, lane * 32, kKvAtomBytes);
            uint8_t* d1 = kv_tile + sw128_offset(key, lane * 32 + 16, kKvAtomBytes);
            *reinterpret_cast<uint4*>(d0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            *reinterpret_cast<uint4*>(d1) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            if (lane < 8)
              *reinterpret_cast<uint4*>(kv_tile + sw128_offset(key, kDimLatent * 2 + lane * 16, kKvAtomBytes)) = rope[jj];
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&kv_full));
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc(128, kMlaHeads, kFmtBF16, kFmtBF16, 0, 0);
      constexpr uint32_t idesc_o = make_idesc(128, kMlaHeads, kFmtBF16, kFmtBF16, 1, 0);
      const uint32_t kv0 = smem_u32(kv_tile);
      int seg = -1;
      for (int i = 0; i < n_mine; ++i) {
        const ChunkPos cp = chunk_pos(i);
        if (cp.first) ++seg;
        const int qb = seg & 1, sb = i & 1;
        const uint32_t ph2 = (i >> 1) & 1;
        if (!mbar_wait(smem_u32(&kv_full), i & 1, &abort_flag, A.err)) break;
        if (cp.first && !mbar_wait(smem_u32(&q_full[qb]), (seg >> 1) & 1, &abort_flag, A.err)) break;
        if (!mbar_wait(smem_u32(&s_empty[sb]), ph2 ^ 1, &abort_flag, A.err)) break;
        tc_fence_after();
        const uint32_t q0 = smem_u32(q_buf + qb * kQBufBytes);
#pragma unroll 1
        for (int a = 0; a < 9; ++a) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc(kv0 + a * kKvAtomBytes + kk * 32, 0, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(q0 + a * kQAtomBytes + kk * 32, 0, 1024, kSwizzle128B);
            mma_f16_ss(tmem_s + sb * 16, ad, bd, idesc_s, (a | kk) != 0);
          }
        }
        mma_commit(smem_u32(&s_full[sb]));
        if (cp.last) mma_commit(smem_u32(&q_empty[qb]));
        if (!mbar_wait(smem_u32(&p_full[sb]), ph2, &abort_flag, A.err)) break;
        if (!mbar_wait(smem_u32(&o_empty[sb]), ph2 ^ 1, &abort_flag, A.err)) break;
        tc_fence_after();
        const uint32_t p0 = smem_u32(p_buf + sb * kPBufBytes);
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t ad = smem_desc(kv0 + 2 * mb * kKvAtomBytes + ks * 2048, kKvAtomBytes, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(p0 + (ks >> 2) * kQAtomBytes + (ks & 3) * 32, 0, 1024, kSwizzle128B);
            mma_f16_ss(tmem_o + sb * 64 + mb * 16, ad, bd, idesc_o, ks != 0);
          }
        }
        mma_commit(smem_u32(&o_full[sb]));
        mma_commit(smem_u32(&p_empty[sb]));
        mma_commit(smem_u32(&kv_empty));
      }
    }
  } else {
    // ================================================================ softmax warps 0-3
    GroupSync gs{smem_u32(&grp_bar), 0};
    int red_i = 0;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float neg_inf = -__int_as_float(0x7f800000);
    float m[kMlaHeads], l[kMlaHeads], o[4][kMlaHeads];
    for (int i = 0; i < n_mine; ++i) {
      const ChunkPos cp = chunk_pos(i);
      const int sb = i & 1;
      const uint32_t ph2 = (i >> 1) & 1;
      if (cp.first) {
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) {
          m[h] = neg_inf; l[h] = 0.f;
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) o[mb][h] = 0.f;
        }
      }
      // validity of this thread's key (same test as the producers)
      const QueryInfo qi = query_info(g, cp.t);
      const int e = cp.cq * kMlaKeys + tid;
      bool valid = false;
      if (qi.ok && e < A.k) {
        const int s = __ldg(A.idx + (int64_t)cp.t * A.k + e);
        valid = s >= 0 && s < qi.len && physical_row(g, qi.b, s) >= 0;
      }
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
      for (int h = 0; h < kMlaHeads; ++h) {
        z[h] = valid ? z[h] * A.scale_log2 : neg_inf;
        const float wm = warp_max(z[h]);
        if (lane == 0) red[red_i][warp][h] = wm;
      }
      if (!gs.sync(&abort_flag, A.err)) break;
      float alpha[kMlaHeads];
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h) {
        const float cm = fmaxf(fmaxf(red[red_i][0][h], red[red_i][1][h]), fmaxf(red[red_i][2][h], red[red_i][3][h]));
        const float mn = fmaxf(m[h], cm);
        alpha[h] = (mn == neg_inf) ? 1.f : exp2f(m[h] - mn);
        z[h] = (z[h] == neg_inf) ? 0.f : exp2f(z[h] - mn);   // z now holds p
        l[h] = l[h] * alpha[h] + z[h];
        m[h] = mn;
      }
      red_i ^= 1;
      // P^T (K-major: row = head, 128 keys = 2 atoms) for the second MMA
      if (!mbar_wait(smem_u32(&p_empty[sb]), ph2 ^ 1, &abort_flag, A.err)) break;
      uint8_t* pb = p_buf + sb * kPBufBytes;
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h)
        *reinterpret_cast<__nv_bfloat16*>(pb + sw128_offset(h, tid * 2, kQAtomBytes)) = __float2bfloat16_rn(z[h]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full[sb]));
      // add this chunk's O^T (lane = latent column within a 128-block)
      if (!mbar_wait(smem_u32(&o_full[sb]), ph2, &abort_flag, A.err)) break;
      tc_fence_after();
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
        float ov[16];
        tmem_ld16(tmem_o + sb * 64 + mb * 16 + lane_off, ov);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) o[mb][h] = fmaf(o[mb][h], alpha[h], ov[h]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&o_empty[sb]));

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
        const int64_t c_first = split_owner((int64_t)cp.t * A.C, A.n_chunks, G);
        const int64_t c_last = split_owner((int64_t)cp.t * A.C + A.C - 1, A.n_chunks, G);
        const int hbase = hg * kMlaHeads;
        if (c_first == c_last) {
#pragma unroll
          for (int h = 0; h < kMlaHeads; ++h) {
            if (h >= h_eff) break;
            const float inv = lt[h] > 0.f ? 1.f / lt[h] : 0.f;
            __nv_bfloat16* orow = A.out + ((int64_t)cp.t * A.H + hbase + h) * kDimLatent;
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) orow[mb * 128 + tid] = __float2bfloat16_rn(o[mb][h] * inv);
            if (A.lse && tid == h)
              A.lse[(int64_t)cp.t * A.H + hbase + h] = lt[h] > 0.f ? (m[h] + log2f(lt[h])) * kLn2 : -__int_as_float(0x7f800000);
          }
        } else {
          const int64_t seg_id = (int64_t)cp.t + blockIdx.x;
#pragma unroll
          for (int h = 0; h < kMlaHeads; ++h) {
            if (h >= h_eff) break;
            const int64_t r = seg_id * A.H + hbase + h;
            float* orow = A.o_part + r * kDimLatent;
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) orow[mb * 128 + tid] = o[mb][h];
            if (tid == h) { A.ml_part[2 * r] = m[h]; A.ml_part[2 * r + 1] = lt[h]; }
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
