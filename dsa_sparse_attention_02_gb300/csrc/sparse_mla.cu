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
// evenly over a persistent grid of two-CTA clusters. The two CTAs of a cluster
// walk the same chunks and split every selected row by columns: CTA r holds
// latent columns 256r..256r+255 (two "pairs" of 64-column atoms) and RoPE
// columns 512+32r..512+32r+31, i.e. half of each 1152-byte row. Each CTA's share
// of a chunk (72 KB) is small enough that two chunks are resident at once, so the
// next chunk streams in while the current one is scored and reduced.
//   * a resolver warp maps each chunk's 128 logical positions to physical cache
//     rows through the block table (-1 for padding or out-of-range entries) up
//     to four chunks ahead, into a shared-memory row table.
//   * four producer warps copy the CTA's columns of the rows with 16-byte
//     cp.async into 128-byte-swizzled K-major atoms (zero-fill for padding), and
//     end each slot with cp.async.mbarrier.arrive.noinc, so a slot's full barrier
//     completes when its copies have landed. e4m3 or int8 cache (mlx-lm "GLM-5.2
//     (glm_moe_dsa) inference": int8 MLA latent KV, dequantized on read): the latent
//     codes are loaded, dequantized (code * per-128 scale) to bf16 and stored instead.
//   * one MMA thread (issuing S steps and PVs as they become ready, so that
//     S(i+1) overlaps the softmax of chunk i): partial S^T = KV . Q^T over the CTA's 288 columns on
//     tcgen05 (M = 128 keys, N = 16 heads) into TMEM, then, once P is known,
//     O^T = V^T . P^T for the CTA's 256 latent columns (M = 128 columns x 2
//     blocks, N = 16, K = 128 keys), V^T read MN-major from the pair slots.
//   * 4 softmax warps (TMEM lane = key) exchange the partial scores with the
//     other CTA through distributed shared memory (8 KB per chunk each way), add
//     them (the same sum in both CTAs, since fp32 addition commutes), and run the
//     online softmax per head in the exp2 domain; both CTAs obtain bit-identical
//     P and statistics. O^T accumulates in TMEM across a query's chunks. The
//     reference max moves only when a chunk's max exceeds it by more than 2^8
//     (p <= 256 otherwise); then the softmax warps wait for PV(i-1) and rescale
//     O in TMEM before releasing P. The partial scores go out with st.async,
//     counted on the receiver's mbarrier; buffer release is a plain signal.
// A cluster that holds every chunk of a query writes the final bf16 output (each
// CTA its 256 columns); other segments write (unnormalized O, running max, sum)
// partials that the combine kernel merges with log-sum-exp weights.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include "kernels.cuh"

namespace dsa {

constexpr int kMlaHeads = 16;                       // heads per CTA (MMA N)
constexpr int kMlaKeys = 128;                       // keys per chunk (MMA M)
constexpr int kMlaKeysC = kMlaKeys;
constexpr int kAtomBytes = kMlaKeys * 128;          // 16 KB: 128 rows x 64 bf16
constexpr int kPairBytes = 2 * kAtomBytes;          // 32 KB
// bf16 cache: five pair slots (two and a half chunks of the CTA's two pairs) that the
// rows are gathered into. Record caches (e4m3 / int8 codes): four bf16 pair slots (two
// chunks) that the codes are converted into, so that a chunk's conversion waits only on
// the attention of the chunk two before it, fed by three code stages of one pair each
// (the pair's 128 codes and one scale of each of the chunk's 128 rows), so that the
// code bytes in flight do not wait on the bf16 slots. Two P buffers (P(i) is written
// once PV(i-2) has released its buffer, without waiting for PV(i-1)); to fit, record
// caches keep one partial-score exchange buffer.
template <int kKv> constexpr int kPairSlotsOf = kKv == kKvBf16 ? 5 : 4;
template <int kKv> constexpr int kPBufsOf = 2;
template <int kKv> constexpr int kXBufsOf = kKv == kKvBf16 ? 2 : 1;
constexpr int kCodeStages = 3;
constexpr int kCodeRowBytes = 128;                          // one pair's codes of a row
constexpr int kCodeBytes = kMlaKeysC * kCodeRowBytes;       // 16 KB
constexpr int kCodeStageBytes = kCodeBytes + kMlaKeysC * 4;   // + the pair's fp32 scale per row
constexpr int kRopeSlots = 2;                       // halves of one RoPE atom (chunk parity)
constexpr int kQAtomBytes = kMlaHeads * 128;        // 2 KB
constexpr int kQAtoms = 6;                          // the CTA's 4 latent atoms + 2 RoPE atoms
constexpr int kQBufBytes = kQAtoms * kQAtomBytes;   // 12 KB
constexpr int kPBufBytes = 2 * kQAtomBytes;         // P^T: 16 heads x 128 keys bf16 = 4 KB
constexpr int kXBufBytes = kMlaKeys * kMlaHeads * 4;  // partial scores from the other CTA: 8 KB
template <int kKv>
constexpr int kMlaSmemBytesOf = 1024 + kPairSlotsOf<kKv> * kPairBytes + (kKv == kKvBf16 ? 0 : kCodeStages * kCodeStageBytes) +
                                kAtomBytes + kQBufBytes + kPBufsOf<kKv> * kPBufBytes + kXBufsOf<kKv> * kXBufBytes;
constexpr int kMlaSmemBytes = kMlaSmemBytesOf<kKvBf16>;
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
constexpr int kMlaTmemCols = 64;                    // S: 2 x 16, O: 2 x 16
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

// Four latent codes (byte i of w = code i) -> fp32 values, exact.
//   e4m3: every e4m3 value (subnormals, the NaN code) is a half value, so the
//   hardware's e4m3x2 -> f16x2 conversion followed by f16 -> f32 is exact;
//   int8: the biased byte x + 128 placed in the mantissa of 2^23 gives the float
//   2^23 + 128 + x exactly, and subtracting 2^23 + 128 leaves x.
template <int kKv>
__device__ __forceinline__ void codes4_to_f32(uint32_t w, float (&f)[4]) {
  if (kKv == kKvInt8) {
    const uint32_t x = w ^ 0x80808080u;
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540u + i)) - 8388736.f;
  } else {
    const float2 a = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3)));
    const float2 b = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3)));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  }
}

// Sixteen latent codes (byte i of word j of c = code 4j+i) times sc, rounded to bf16
// and packed in pairs: pk[k] = (bf16(code[2k] * sc), bf16(code[2k+1] * sc)), the
// exact code times sc rounded once to fp32, then to bf16. (An integer construction of
// the e4m3 values measured 40% slower than the hardware conversion on this part.)
template <int kKv>
__device__ __forceinline__ void dequant16(const uint4 c, float sc, uint32_t (&pk)[8]) {
  const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
  const float2 s2 = make_float2(sc, sc);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float f[4];
    codes4_to_f32<kKv>(w4[j], f);
    // two products per packed fp32x2 multiply (each rounded as a single multiply)
    const float2 lo = __fmul2_rn(make_float2(f[0], f[1]), s2), hi = __fmul2_rn(make_float2(f[2], f[3]), s2);
    pk[2 * j] = pack_bf16x2(lo.x, lo.y);
    pk[2 * j + 1] = pack_bf16x2(hi.x, hi.y);
  }
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

template <int kKv>
__global__ void __launch_bounds__(kMlaThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap map_q, const MlaArgs A) {
  constexpr bool kRecord = kKv != kKvBf16;   // 656-byte records: codes, scales, RoPE
  constexpr int kPairSlots = kPairSlotsOf<kKv>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // Swizzled operand tiles first (each 1024-byte aligned), then the record caches' code
  // stages, which cp.async and plain loads address at 16-byte granularity.
  uint8_t* pair_buf = smem;                                         // kPairSlots x 32 KB
  uint8_t* rope_buf = pair_buf + kPairSlots * kPairBytes;           // 16 KB
  uint8_t* q_buf = rope_buf + kAtomBytes;                           // 12 KB
  uint8_t* p_buf = q_buf + kQBufBytes;                              // 2 x 4 KB
  constexpr int kPBufs = kPBufsOf<kKv>, kXBufs = kXBufsOf<kKv>;
  float4* x_buf = reinterpret_cast<float4*>(p_buf + kPBufs * kPBufBytes);  // kXBufs x [4 head quads][128 keys]
  uint8_t* code_buf = reinterpret_cast<uint8_t*>(x_buf) + kXBufs * kXBufBytes;   // record caches: kCodeStages x 16.5 KB

  __shared__ uint64_t pair_full[kPairSlots], pair_empty[kPairSlots], rope_full[kRopeSlots], rope_empty[kRopeSlots];
  __shared__ uint64_t q_full, q_empty;
  __shared__ uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2], o_full[2], o_free, grp_bar;
  __shared__ uint64_t x_full[2], x_free[2];   // partial-score exchange with the other CTA
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  __shared__ __align__(16) float red[2][4][kMlaHeads];
  __shared__ __align__(16) int over_s[2][4];   // per softmax warp: a key exceeds the reference by > 2^8
  __shared__ __align__(16) int rows_s[kRowBufs][kMlaKeys];   // physical row per key of a chunk, -1 = none
  __shared__ uint64_t rows_full[kRowBufs], rows_empty[kRowBufs];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GeomDev& g = A.g;
  const int rank = (int)cluster_ctarank();            // column half of this CTA
  const int peer = rank ^ 1;
  const int G = (int)cluster_count_x();               // clusters (work splits over clusters)
  const int cid = (int)cluster_id_x();
  const int hg = blockIdx.y;
  const int h_eff = min(kMlaHeads, A.H - hg * kMlaHeads);
  const int64_t c_begin = split_begin(cid, A.n_chunks, G);
  const int64_t c_end = split_begin(cid + 1, A.n_chunks, G);
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
  // The same walked one chunk at a time, without a division per step.
  auto chunk_next = [&](ChunkPos& cp, int i_next) {
    ++cp.chunk;
    if (++cp.cq == A.C) { cp.cq = 0; ++cp.t; }
    cp.first = (cp.cq == 0);
    cp.last = (i_next == n_mine - 1) || (cp.cq == A.C - 1);
  };
  // Q atoms of this CTA: latent columns 256*rank + 64a (a = 0..3); then two RoPE
  // atoms. The CTA's RoPE columns 32*rank..32*rank+31 sit in 16-byte chunks
  // 4p..4p+3 of the KV RoPE atom for chunk parity p, and must sit at the same
  // chunks of the Q atom the MMA pairs them with: atom 4 starts at column 512
  // (its chunks 4*rank.. hold them), atom 5 at 480 + 64*rank (its chunks
  // 4*(1-rank).. hold them; columns past 575 are zero-filled by TMA).
  auto load_q = [&](int t) {
    const uint32_t bar = smem_u32(&q_full);
    mbar_arrive_expect_tx(bar, kQAtoms * h_eff * 128);   // out-of-range columns are zero-filled and counted
    for (int a = 0; a < kQAtoms; ++a)
      tma_load_2d(smem_u32(q_buf + a * kQAtomBytes), &map_q, bar,
                  a < 4 ? 256 * rank + 64 * a : (a == 4 ? kDimLatent : kDimLatent - 32 + 64 * rank),
                  t * A.H + hg * kMlaHeads);
  };

  if (tid == 0) {
    abort_flag = 0;
    // bf16: a pair slot is filled by the cp.async copies of 64 producer threads (noinc
    // arrivals); records: by the conversions of all 128 producer threads
    for (int j = 0; j < kPairSlots; ++j) {
      mbar_init(smem_u32(&pair_full[j]), kRecord ? slot_producers : 64);
      mbar_init(smem_u32(&pair_empty[j]), 1);
    }
    for (int j = 0; j < kRopeSlots; ++j) { mbar_init(smem_u32(&rope_full[j]), slot_producers); mbar_init(smem_u32(&rope_empty[j]), 1); }
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&q_empty), 1);
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_u32(&s_full[j]), 1);
      mbar_init(smem_u32(&s_empty[j]), 4);
      mbar_init(smem_u32(&p_full[j]), 4);
      mbar_init(smem_u32(&p_empty[j]), 1);
      mbar_init(smem_u32(&x_full[j]), 1);     // local expect_tx + 8 KB of st.async from the other CTA
      mbar_init(smem_u32(&x_free[j]), 4);     // one signal per softmax warp of the other CTA
    }
    mbar_init(smem_u32(&o_full[0]), 1);  // one phase per even chunk's PV
    mbar_init(smem_u32(&o_full[1]), 1);  // and per odd chunk's
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
  // The other CTA's barriers are initialized before any remote arrival.
  cluster_sync();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tmem_s = tmem;          // + 16 * buf
  const uint32_t tmem_o = tmem + 32;     // + 16 * block
  // The query rows are inputs of this call, not results of the preceding kernel.
  if (warp == kProdWarp0 && lane == 0 && n_mine > 0) { tma_prefetch_desc(&map_q); load_q(chunk_pos(0).t); }
  // Only the resolver reads what the preceding kernel wrote (the index rows); it
  // waits for that kernel (griddepcontrol.wait) before its first index load, and
  // every other role depends on the resolver's row table.

  if (warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps && !kRecord) {
    // ================================================================ producers (bf16 cache)
    // Two groups of two warps: group jl (warps 4-5: jl = 0; warps 6-7: jl = 1) fills
    // latent pair jl of every chunk, so that both pairs of a chunk are requested at
    // once; warp wg of a group copies rows [64*wg, 64*wg+64) of the pair. Every
    // producer warp also copies the RoPE columns of rows [32*pw, 32*pw+32). 16-byte
    // cp.async (zero-fill for padding), slot completion through
    // cp.async.mbarrier.arrive.noinc.
    const int pw = warp - kProdWarp0;
    const int jl = pw >> 1, wg = pw & 1;
    const int j = 2 * rank + jl;                 // pair of the row: latent columns 128j..128j+127
    int seg = 0;
    // warp-uniform bounded wait
    auto slot_acquire = [&](uint32_t bar, uint32_t parity) -> bool {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(bar, parity, &abort_flag, A.err) ? 1 : 0;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    const size_t row_bytes = (size_t)(kDimQK * 2);
    const size_t rope_off = (size_t)(kDimLatent * 2) + 64 * rank;
    ChunkPos cp = chunk_pos(0);
    for (int i = 0; i < n_mine; chunk_next(cp, ++i)) {
      if (cp.first) {
        if (pw == 0 && seg > 0) {
          if (!slot_acquire(smem_u32(&q_empty), (seg & 1) ^ 1)) break;
          if (lane == 0) load_q(cp.t);
        }
        ++seg;
      }
      const int rb = i % kRowBufs, rs = i % kRopeSlots;
      if (!slot_acquire(smem_u32(&rows_full[rb]), (i / kRowBufs) & 1)) break;
      mbar_try_wait(smem_u32(&rows_full[rb]), (i / kRowBufs) & 1);   // acquire in every lane (phase is complete)
      const int* rows = rows_s[rb];
      const uint8_t* kv = A.kv;
      // RoPE columns of this CTA: 4 lanes per row (64 B), 8 rows per instruction,
      // into logical 16-byte chunks 4*rs..4*rs+3 of the shared RoPE atom's rows
      if (!slot_acquire(smem_u32(&rope_empty[rs]), ((i / kRopeSlots) & 1) ^ 1)) break;
      {
        const uint32_t dst0 = smem_u32(rope_buf);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ri = 32 * pw + 8 * q + (lane >> 2);
          const int row = rows[ri];
          const int cb = (lane & 3) * 16;
          cp_async_16(dst0 + sw128_offset(ri, 64 * rs + cb, 0),
                      kv + (int64_t)(row >= 0 ? row : 0) * row_bytes + rope_off + cb, row >= 0 ? 16u : 0u);
        }
        cp_async_arrive_noinc(smem_u32(&rope_full[rs]));
      }
      const int gidx = 2 * i + jl, ps = gidx % kPairSlots;
      if (!slot_acquire(smem_u32(&pair_empty[ps]), ((gidx / kPairSlots) & 1) ^ 1)) break;
      uint8_t* slot = pair_buf + ps * kPairBytes;
      // 16 lanes per row (256 B of the pair), 2 rows per instruction: lane half h
      // takes rows r0 .. r0+31, r0 = 64*wg + 32*h, whose indices it reads up front
      const int r0 = 64 * wg + 32 * (lane >> 4);
      const int cb = (lane & 15) * 16;
      int rr[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int4 v = *reinterpret_cast<const int4*>(rows + r0 + 4 * q);
        rr[4 * q] = v.x; rr[4 * q + 1] = v.y; rr[4 * q + 2] = v.z; rr[4 * q + 3] = v.w;
      }
      const uint32_t dst0 = smem_u32(slot);
      const uint8_t* src0 = kv + j * 256 + cb;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int row = rr[jj];
        cp_async_16(dst0 + sw128_offset(r0 + jj, cb, kAtomBytes), src0 + (int64_t)(row >= 0 ? row : 0) * row_bytes,
                    row >= 0 ? 16u : 0u);
      }
      cp_async_arrive_noinc(smem_u32(&pair_full[ps]));
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&rows_empty[rb]));
    }
  } else if (warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps) {
    // ================================================================ producers (record caches)
    // Pair g = 2i + jl is latent pair jl of chunk i (this CTA's latent group 2*rank+jl).
    // Warp pw owns rows [32*pw, 32*pw+32) of every chunk. Step g: the warp copies its
    // rows' 128 codes and one scale of pair g into code stage g % 3 (16-byte and 4-byte
    // cp.async, zero-fill for padding, one commit group per step), and, with a new
    // chunk, its rows' RoPE columns into the RoPE atom; then it converts pair g - 2 of
    // the same rows, code * scale rounded to bf16, into pair slot (g - 2) % 4 (the
    // swizzled K-major layout the MMA reads) and marks its share of the slot full. Two
    // pairs are thus in flight while one is converted, and a pair's slot is the one
    // pair g - 6 used, freed by the attention of the chunk two before: the conversion
    // never waits on the chunk just before it. Every wait before converting pair g - 2
    // depends only on pairs before it (the query buffer of a new segment, which the MMA
    // frees after the previous chunk's scores, is taken after that chunk's conversion).
    constexpr int kLag = 2;
    const int pw = warp - kProdWarp0;
    auto slot_acquire = [&](uint32_t bar, uint32_t parity) -> bool {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(bar, parity, &abort_flag, A.err) ? 1 : 0;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    const uint8_t* kv = A.kv;
    // A warp's rows of a code stage are copied and read by that warp alone, so the
    // stages need no barrier: cp.async groups (one per step) say when a pair's copies
    // have landed, and the warp's own order says when a stage may be reused.
    auto convert = [&](int gc, int pending) -> bool {
      const int cs = gc % kCodeStages, ps = gc % kPairSlots;
      if (pending >= 2) cp_async_wait<2>();
      else if (pending == 1) cp_async_wait<1>();
      else cp_async_wait<0>();
      __syncwarp();   // the row's scale was copied by another lane of the warp
      if (!slot_acquire(smem_u32(&pair_empty[ps]), ((gc / kPairSlots) & 1) ^ 1)) return false;
      const uint8_t* stg = code_buf + cs * kCodeStageBytes;
      const float* scl = reinterpret_cast<const float*>(stg + kCodeBytes);   // [128 rows]
      uint8_t* slot = pair_buf + ps * kPairBytes;
      // A quarter warp converts rows r0 (even) and r0+1 together: lanes 0-3 of it take
      // pieces p = 4a + (0..3) of row r0 and lanes 4-7 pieces 4(1-a) + (0..3) of row
      // r0+1. With the stage and the slot both swizzled by row, the eight lanes then
      // touch eight different 16-byte bank groups on every load and store.
      const int rsel = (lane >> 2) & 1, p4 = lane & 3;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        const int r = 32 * pw + 8 * q + 2 * (lane >> 3) + rsel;
        const float sc = scl[r];
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          const int piece = 4 * (a ^ rsel) + p4;   // codes 16*piece .. 16*piece+15 of the pair
          const uint4 c = *reinterpret_cast<const uint4*>(stg + r * kCodeRowBytes + ((piece ^ (r & 7)) << 4));
          uint32_t pk[8];
          dequant16<kKv>(c, sc, pk);
          *reinterpret_cast<uint4*>(slot + sw128_offset(r, 32 * piece, kAtomBytes)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(slot + sw128_offset(r, 32 * piece + 16, kAtomBytes)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      fence_proxy_async_smem();   // the MMA reads the slot through the async proxy
      mbar_arrive(smem_u32(&pair_full[ps]));
      return true;
    };
    int seg = 1;   // segments whose query has been loaded (the first at the kernel's start)
    bool ok = true;
    const int n_pairs = 2 * n_mine;
    ChunkPos cp = chunk_pos(0);
    for (int g = 0; g < n_pairs + kLag && ok; ++g) {
      if (g < n_pairs) {
        const int i = g >> 1, jl = g & 1, rb = i % kRowBufs, cs = g % kCodeStages;
        if (!slot_acquire(smem_u32(&rows_full[rb]), (i / kRowBufs) & 1)) break;
        mbar_try_wait(smem_u32(&rows_full[rb]), (i / kRowBufs) & 1);   // acquire in every lane (phase is complete)
        const int* rows = rows_s[rb];
        __syncwarp();   // every lane has read this stage's previous pair (converted two steps ago)
        {
          uint8_t* stg = code_buf + cs * kCodeStageBytes;
          const uint32_t dst_codes = smem_u32(stg), dst_scales = smem_u32(stg + kCodeBytes);
          const int part = lane & 7;
          const int64_t col = 256 * rank + 128 * jl + 16 * part;
#pragma unroll
          for (int q = 0; q < 8; ++q) {   // 8 lanes per row (128 B), 4 rows per instruction; piece swizzled by row
            const int r = 32 * pw + 4 * q + (lane >> 3);
            const int row = rows[r];
            cp_async_16(dst_codes + r * kCodeRowBytes + ((part ^ (r & 7)) << 4), kv + rec_codes_at(row >= 0 ? row : 0) + col,
                        row >= 0 ? 16u : 0u);
          }
          const int r = 32 * pw + lane;
          const int row = rows[r];
          cp_async_4(dst_scales + 4 * r, kv + rec_scales_at(row >= 0 ? row : 0) + 4 * (2 * rank + jl),
                     row >= 0 ? 4u : 0u);
          cp_async_commit();
        }
        // the RoPE copies after the codes: their slot frees only once the chunk two
        // before has been scored, which the codes need not wait for
        if (jl == 0) {
          const int rs = i % kRopeSlots;
          if (!slot_acquire(smem_u32(&rope_empty[rs]), ((i / kRopeSlots) & 1) ^ 1)) break;
          const uint32_t dst0 = smem_u32(rope_buf);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int ri = 32 * pw + 8 * q + (lane >> 2);
            const int row = rows[ri];
            const int cb = (lane & 3) * 16;
            cp_async_16(dst0 + sw128_offset(ri, 64 * rs + cb, 0),
                        kv + rec_rope_at(row >= 0 ? row : 0) + 64 * rank + cb, row >= 0 ? 16u : 0u);
          }
          cp_async_arrive_noinc(smem_u32(&rope_full[rs]));
        }
        if (jl == 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&rows_empty[rb]));   // the copies need no row ids any more
        }
      }
      if (g >= kLag) {
        const int gc = g - kLag;
        // groups committed after pair gc's: pairs gc+1 .. min(g, n_pairs-1)
        if (!convert(gc, (g < n_pairs ? g : n_pairs - 1) - gc)) { ok = false; break; }
        if (gc & 1) {
          // chunk gc/2 is converted; a new segment's query follows once the MMA has
          // freed the buffer after the previous segment's last scores
          const int ic = gc >> 1;
          if (ic + 1 < n_mine) {
            chunk_next(cp, ic + 1);
            if (cp.first) {
              if (pw == 0) {
                if (!slot_acquire(smem_u32(&q_empty), (seg & 1) ^ 1)) break;
                if (lane == 0) load_q(cp.t);
              }
              ++seg;
            }
          }
        }
      }
    }
  } else if (warp == kResolverWarp) {
    // ================================================================ row resolver
    ChunkPos cp = chunk_pos(0);
    // the request geometry is an input of the call: looked up before the wait
    QueryInfo qi = query_info_warp(g, cp.t);
    int t_cached = cp.t;
    griddep_wait();
    for (int i = 0; i < n_mine; chunk_next(cp, ++i)) {
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
    // Issues, in order within each kind, the S steps of chunk s_i (RoPE, pair 0,
    // pair 1 as each lands) and the PV of chunk pv_i < s_i (once its P is
    // written), whichever is ready first, so that S(i+1) overlaps softmax(i) and
    // PV(i) never waits behind the next chunk's loads. A PV is preferred when both
    // are ready, since it releases ring slots.
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc(128, kMlaHeads, kFmtBF16, kFmtBF16, 0, 0);
      constexpr uint32_t idesc_o = make_idesc(128, kMlaHeads, kFmtBF16, kFmtBF16, 1, 0);
      // descriptors built once; each MMA offsets them by a byte distance
      const uint64_t dk_pair = smem_desc(smem_u32(pair_buf), 0, 1024, kSwizzle128B);            // K-major (S)
      const uint64_t dmn_pair = smem_desc(smem_u32(pair_buf), kAtomBytes, 1024, kSwizzle128B);  // MN-major (PV)
      const uint64_t dk_rope = smem_desc(smem_u32(rope_buf), 0, 1024, kSwizzle128B);
      const uint64_t dk_q = smem_desc(smem_u32(q_buf), 0, 1024, kSwizzle128B);
      const uint64_t dk_p = smem_desc(smem_u32(p_buf), 0, 1024, kSwizzle128B);
      int s_i = 0, s_step = 0, s_seg = -1;   // s_step: 0 = RoPE next, 1 = pair 0 next, 2 = pair 1 next
      int pv_i = 0, pv_seg = -1;
      ChunkPos s_cp = chunk_pos(0), pv_cp = s_cp;
      uint64_t t_idle = globaltimer_ns();
      while (pv_i < n_mine) {
        bool progress = false;
        if (pv_i < s_i) {
          const ChunkPos& cp = pv_cp;
          const int sb = pv_i % kPBufs;
          // a new segment's first PV overwrites O: the previous segment's O must have been read
          const bool o_ok = !cp.first || pv_seg < 0 || mbar_test_wait(smem_u32(&o_free), pv_seg & 1);
          if (o_ok && mbar_test_wait(smem_u32(&p_full[sb]), (pv_i / kPBufs) & 1)) {
            if (cp.first) ++pv_seg;
            tc_fence_after();
            const uint64_t bd0 = desc_add(dk_p, sb * kPBufBytes);
#pragma unroll
            for (int mb = 0; mb < 2; ++mb) {
              const int ps = (2 * pv_i + mb) % kPairSlots;
              const uint64_t ad0 = desc_add(dmn_pair, ps * kPairBytes);
#pragma unroll
              for (int ks = 0; ks < 8; ++ks)
                mma_f16_ss(tmem_o + mb * 16, desc_add(ad0, ks * 2048),
                           desc_add(bd0, (ks >> 2) * kQAtomBytes + (ks & 3) * 32), idesc_o,
                           (ks != 0 || !cp.first) ? 1u : 0u);
              mma_commit(smem_u32(&pair_empty[ps]));
            }
            mma_commit(smem_u32(&o_full[pv_i & 1]));
            mma_commit(smem_u32(&p_empty[sb]));
            chunk_next(pv_cp, ++pv_i);
            progress = true;
          }
        }
        if (s_i < n_mine) {
          const ChunkPos& cp = s_cp;
          const int sb = s_i & 1, rs = s_i % kRopeSlots;
          const uint32_t d_s = tmem_s + sb * 16;
          if (s_step == 0) {
            if ((!cp.first || mbar_test_wait(smem_u32(&q_full), (s_seg + 1) & 1)) &&
                mbar_test_wait(smem_u32(&s_empty[sb]), ((s_i >> 1) & 1) ^ 1) &&
                mbar_test_wait(smem_u32(&rope_full[rs]), (s_i / kRopeSlots) & 1)) {
              if (cp.first) ++s_seg;
              fence_proxy_async_smem();   // slot filled through the generic proxy (cp.async / st.shared)
              tc_fence_after();
              // RoPE columns 32*rank..32*rank+31: K-steps 2*rs and 2*rs+1 of the atom,
              // against the Q RoPE atom that holds the same columns at the same chunks
              const uint64_t q_rope = desc_add(dk_q, (rs == rank ? 4 : 5) * kQAtomBytes);
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                const uint32_t off = (2 * rs + kk) * 32;
                mma_f16_ss(d_s, desc_add(dk_rope, off), desc_add(q_rope, off), idesc_s, kk != 0);
              }
              mma_commit(smem_u32(&rope_empty[rs]));
              s_step = 1;
              progress = true;
            }
          } else {
            const int jl = s_step - 1, gidx = 2 * s_i + jl, ps = gidx % kPairSlots;
            if (mbar_test_wait(smem_u32(&pair_full[ps]), (gidx / kPairSlots) & 1)) {
              fence_proxy_async_smem();
              tc_fence_after();
              const uint64_t a0 = desc_add(dk_pair, ps * kPairBytes);
              const uint64_t b0 = desc_add(dk_q, 2 * jl * kQAtomBytes);
#pragma unroll
              for (int a2 = 0; a2 < 2; ++a2) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_f16_ss(d_s, desc_add(a0, a2 * kAtomBytes + kk * 32), desc_add(b0, a2 * kQAtomBytes + kk * 32),
                             idesc_s, 1);
              }
              if (jl == 1) {
                mma_commit(smem_u32(&s_full[sb]));
                if (cp.last) mma_commit(smem_u32(&q_empty));
                chunk_next(s_cp, ++s_i);
                s_step = 0;
              } else {
                s_step = 2;
              }
              progress = true;
            }
          }
        }
        if (progress) {
          t_idle = globaltimer_ns();
        } else {
          if (abort_flag) break;
          if (globaltimer_ns() - t_idle > kWaitLimitNs) {
            abort_flag = 1;
            record_error(A.err, kDevTimeout);
            break;
          }
        }
      }
    }
  } else if (warp < 4) {
    // ================================================================ softmax warps 0-3
    GroupSync gs{smem_u32(&grp_bar), 0};
    int red_i = 0;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float neg_inf = -__int_as_float(0x7f800000);
    float m[kMlaHeads], l[kMlaHeads];
    // exchange addresses: this thread's float4 slot per head quad, locally and in the other CTA
    const uint32_t x_local = smem_u32(x_buf) + tid * 16;
    const uint32_t x_remote = mapa_shared(x_local, peer);
    const uint32_t xfull_remote = mapa_shared(smem_u32(&x_full[0]), peer);
    const uint32_t xfree_remote = mapa_shared(smem_u32(&x_free[0]), peer);
    ChunkPos cp = chunk_pos(0);
    for (int i = 0; i < n_mine; chunk_next(cp, ++i)) {
      const int sb = i & 1;                          // S buffer in TMEM
      const uint32_t ph2 = (i >> 1) & 1;
      const int xb = i % kXBufs, pbi = i % kPBufs;   // exchange and P buffers
      const uint32_t xph = (i / kXBufs) & 1, pph = (i / kPBufs) & 1;
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
      // ---- exchange the partial scores with the other CTA (buffer sb, layout [quad][key]):
      // st.async into its buffer, counted on its x_full; it signals x_free once read.
      if (!mbar_wait(smem_u32(&x_free[xb]), xph ^ 1, &abort_flag, A.err)) break;   // it has read buffer xb
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        st_async_v4(x_remote + (uint32_t)(xb * kXBufBytes + q4 * kMlaKeys * 16), z[4 * q4], z[4 * q4 + 1],
                    z[4 * q4 + 2], z[4 * q4 + 3], xfull_remote + xb * 8);
      if (tid == 0) mbar_arrive_expect_tx(smem_u32(&x_full[xb]), kXBufBytes);
      if (!mbar_wait<true>(smem_u32(&x_full[xb]), xph, &abort_flag, A.err)) break;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 v = x_buf[xb * (kXBufBytes / 16) + q4 * kMlaKeys + tid];
        z[4 * q4] += v.x; z[4 * q4 + 1] += v.y; z[4 * q4 + 2] += v.z; z[4 * q4 + 3] += v.w;
      }
      __syncwarp();   // the warp's reads of the buffer are done (their sums are in registers)
      if (lane == 0) mbar_arrive_remote_signal(xfree_remote + xb * 8);
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h) z[h] = valid ? z[h] * A.scale_log2 : neg_inf;
      // The reference max of a head moves only where this chunk exceeds it by more
      // than 2^8. Usually no key does: one flag per warp settles that, and only
      // otherwise is the chunk max per head reduced across the 128 keys.
      bool over = false;
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h) over |= z[h] > m[h] + kRescaleLog2;   // also true for m = -inf
      {
        const bool warp_over = __any_sync(0xffffffffu, over);
        if (lane == 0) over_s[red_i][warp] = warp_over ? 1 : 0;
      }
      if (!gs.sync(&abort_flag, A.err)) break;
      const int4 ov4 = *reinterpret_cast<const int4*>(over_s[red_i]);
      red_i ^= 1;
      float alpha[kMlaHeads];
      bool any_raise = false;
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h) alpha[h] = 1.f;
      if (ov4.x | ov4.y | ov4.z | ov4.w) {   // uniform over the four warps
        {
          // after the butterfly, lanes 2h' and 2h'+1 hold the warp max of head hidx below
          // (exchange distances 16, 8, 4, 2 select head bits 3, 2, 1, 0)
          const float wm = warp_max16(z);
          const int hidx = ((lane >> 4) & 1) << 3 | ((lane >> 3) & 1) << 2 | ((lane >> 2) & 1) << 1 | ((lane >> 1) & 1);
          if ((lane & 1) == 0) red[red_i][warp][hidx] = wm;
        }
        if (!gs.sync(&abort_flag, A.err)) break;
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
        red_i ^= 1;
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) {
          const float cm = cmv[h];
          if (cm > m[h] + kRescaleLog2) {       // also true for the first finite max (m = -inf)
            alpha[h] = (m[h] == neg_inf) ? 0.f : fast_exp2(m[h] - cm);
            any_raise = true;
            m[h] = cm;
          }
        }
      }
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h) {
        l[h] *= alpha[h];
        z[h] = (z[h] == neg_inf) ? 0.f : fast_exp2(z[h] - m[h]);   // z now holds p <= 256
        l[h] += z[h];
      }
      // PV(j) completes phase j/2 of o_full[j % 2]. A parity wait is unambiguous while
      // the barrier's previous phase has completed: before P(j) was written, PV(j-2)
      // had completed (P buffer j % 2 was released by it), so a wait for PV(i-1) here
      // or for PV(i) at a segment end never returns on an older phase, and the softmax
      // need not observe every PV. It waits for PV(i-1) only to rescale O, so P(i) no
      // longer waits for the previous chunk's PV.
      if (any_raise && !cp.first) {
        // O in TMEM holds this segment's earlier chunks: once PV(i-1) has completed,
        // scale the raised heads' columns by alpha (PV(i) waits for this chunk's P).
        if (!mbar_wait(smem_u32(&o_full[(i - 1) & 1]), ((i - 1) >> 1) & 1, &abort_flag, A.err)) break;
        tc_fence_after();
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
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
      if (!mbar_wait(smem_u32(&p_empty[pbi]), pph ^ 1, &abort_flag, A.err)) break;
      uint8_t* pb = p_buf + pbi * kPBufBytes;
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h)
        *reinterpret_cast<__nv_bfloat16*>(pb + sw128_offset(h, tid * 2, kQAtomBytes)) = __float2bfloat16_rn(z[h]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full[pbi]));

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
        if (!mbar_wait(smem_u32(&o_full[i & 1]), (i >> 1) & 1, &abort_flag, A.err)) break;
        tc_fence_after();
        const int64_t c_first = split_owner((int64_t)cp.t * A.C, A.n_chunks, G);
        const int64_t c_last = split_owner((int64_t)cp.t * A.C + A.C - 1, A.n_chunks, G);
        const bool whole = c_first == c_last;
        const int hbase = hg * kMlaHeads;
        const int64_t row0 = whole ? (int64_t)cp.t * A.H + hbase : ((int64_t)cp.t + cid) * A.H + hbase;
        const int col0 = 256 * rank + tid;
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) lt[h] = lt[h] > 0.f ? 1.f / lt[h] : 0.f;   // now 1/l
#pragma unroll 1
        for (int mb = 0; mb < 2; ++mb) {
          float ov[16];
          tmem_ld16(tmem_o + mb * 16 + lane_off, ov);
          tmem_ld_wait();
          if (whole) {
            __nv_bfloat16* op = A.out + row0 * kDimLatent + mb * 128 + col0;
#pragma unroll
            for (int h = 0; h < kMlaHeads; ++h)
              if (h < h_eff) op[(int64_t)h * kDimLatent] = __float2bfloat16_rn(ov[h] * lt[h]);
          } else {
            float* op = A.o_part + row0 * kDimLatent + mb * 128 + col0;
#pragma unroll
            for (int h = 0; h < kMlaHeads; ++h)
              if (h < h_eff) op[(int64_t)h * kDimLatent] = ov[h];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&o_free));
        if (rank == 0 && tid < h_eff) {   // the statistics are identical in both CTAs
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

  // The combine kernel may start launching; it waits for this grid to finish.
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  // Neither CTA leaves while the other may still write into its shared memory.
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kMlaTmemCols);
  }
}

// Merge the partial segments of every query that more than one cluster worked on.
__global__ void __launch_bounds__(128) mla_combine_kernel(const MlaArgs A, int G) {
  const int t = blockIdx.x;
  const int h = blockIdx.y;
  const int64_t c_first = split_owner((int64_t)t * A.C, A.n_chunks, G);
  const int64_t c_last = split_owner((int64_t)t * A.C + A.C - 1, A.n_chunks, G);
  if (c_first == c_last) return;
  griddep_wait();   // the partials come from the attention grid just before
  const float neg_inf = -__int_as_float(0x7f800000);
  const float2* ml = reinterpret_cast<const float2*>(A.ml_part);
  // Segments in groups of four, every load of a group issued before any is used; a
  // query of at most four segments (the usual case is two) takes one round of loads.
  float mx = neg_inf, L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  float2 s4[4];
  float o4[4][4];
  auto load4 = [&](int64_t c0, bool rows) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t r = (t + c0 + u) * A.H + h;
      const bool in = c0 + u <= c_last;
      s4[u] = in ? ml[r] : make_float2(neg_inf, 0.f);
      if (rows) {
#pragma unroll
        for (int j = 0; j < 4; ++j) o4[u][j] = in ? A.o_part[r * kDimLatent + j * 128 + threadIdx.x] : 0.f;
      }
    }
  };
  auto add4 = [&]() {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (s4[u].x == neg_inf) continue;   // no valid key in that segment (or past the last)
      const float wgt = exp2f(s4[u].x - mx);
      L = fmaf(wgt, s4[u].y, L);
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] = fmaf(wgt, o4[u][j], acc[j]);
    }
  };
  if (c_last - c_first < 4) {
    load4(c_first, true);
#pragma unroll
    for (int u = 0; u < 4; ++u) mx = fmaxf(mx, s4[u].x);
    add4();
  } else {
    for (int64_t c0 = c_first; c0 <= c_last; c0 += 4) {
      load4(c0, false);
#pragma unroll
      for (int u = 0; u < 4; ++u) mx = fmaxf(mx, s4[u].x);
    }
    for (int64_t c0 = c_first; c0 <= c_last; c0 += 4) {
      load4(c0, true);
      add4();
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* orow = A.out + ((int64_t)t * A.H + h) * kDimLatent;
#pragma unroll
  for (int j = 0; j < 4; ++j) orow[j * 128 + threadIdx.x] = __float2bfloat16_rn(acc[j] * inv);
  if (A.lse && threadIdx.x == 0) A.lse[(int64_t)t * A.H + h] = L > 0.f ? (mx + log2f(L)) * kLn2 : neg_inf;
}

// ------------------------------------------------------------------ host side
// Clusters of two CTAs that can be resident at once (the grid is persistent),
// cached per device; the cluster placement limit can be below half the SM count.
static int mla_max_clusters(int num_sms) {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaFuncSetAttribute(sparse_mla_kernel<kKvBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMlaSmemBytes) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(kMlaThreads, 1, 1);
    cfg.dynamicSmemBytes = kMlaSmemBytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
    cfg.attrs = at; cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_mla_kernel<kKvBf16>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  if (n <= 0 || n > num_sms / 2) n = num_sms / 2;
  if (n < 1) n = 1;
  cache[dev] = n;
  return n;
}

int mla_grid(int64_t n_chunks, int num_sms) {
  const int clusters = mla_max_clusters(num_sms);
  return (int)(n_chunks < clusters ? n_chunks : clusters);
}

size_t mla_partial_bytes(int T, int H, int grid) {
  const size_t rows = (size_t)(T + grid) * H;
  return rows * kDimLatent * sizeof(float) + rows * 2 * sizeof(float);
}

cudaError_t mla_launch(int kv_format, const CUtensorMap& map_q, MlaArgs A, int grid, bool pdl, cudaStream_t st) {
  const int hgroups = (A.H + kMlaHeads - 1) / kMlaHeads;
  auto kern = kv_format == kKvE4m3 ? sparse_mla_kernel<kKvE4m3>
            : kv_format == kKvInt8 ? sparse_mla_kernel<kKvInt8> : sparse_mla_kernel<kKvBf16>;
  const int smem = kv_format == kKvBf16 ? kMlaSmemBytesOf<kKvBf16> : kMlaSmemBytesOf<kKvE4m3>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * grid, hgroups, 1);
  cfg.blockDim = dim3(kMlaThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at; cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, map_q, A);
  if (e != cudaSuccess) return e;
  if (A.C > 1) {  // a query with several chunks may span clusters
    // the shared-memory configuration of the attention grid it follows
    e = cudaFuncSetAttribute(mla_combine_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cc{};
    cc.gridDim = dim3(A.g.T, A.H, 1);
    cc.blockDim = dim3(128, 1, 1);
    cc.stream = st;
    cc.attrs = &at[1]; cc.numAttrs = 1;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    e = cudaLaunchKernelEx(&cc, mla_combine_kernel, A, grid);
  }
  return e;
}

}  // namespace dsa
