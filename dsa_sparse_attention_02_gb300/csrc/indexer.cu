// Lightning-indexer scores on tcgen05 tensor cores.
//
//   I[t,s] = k_scale[s] * sum_h (w[t,h] * q_scale[t,h]) * ReLU(qcode[t,h,:] . kcode[s,:])
//
// which equals sum_h w[t,h] * ReLU(q[t,h,:] . k[s,:]) for dequantized q and k because
// the scales are positive (mlx-lm "GLM-5.2 (glm_moe_dsa) inference", IndexShare
// commit, names the lightning indexer; lmdeploy "feat: support GLM-5.2", Changes).
//
// Work unit = (request b, 128-key tile, group of up to QG queries of b). The key
// tile is the MMA's M side (128 rows = two 64-token pages, read by TMA straight
// from the paged index-key cache), the group's QG x Hp query-head rows are the N
// side (N = QG*Hp <= 256), K = 128 dims (e4m3: kind::f8f6f4, 4 MMAs of K=32;
// bf16: kind::f16, 8 MMAs of K=16). The fp32 accumulator sits in TMEM, one lane
// per key; the epilogue thread of that lane applies ReLU, the per-head weight and
// the head sum within its own registers, multiplies the key's scale and writes
// one score per query, -inf past the query's causal position.
//
// Roles: warp P decodes 32 units at a time (one per lane) and fills an S-stage
// smem ring by TMA: the two key pages, the group's query rows, and by bulk copy
// the pages' key scales and the queries' w and q_scale rows, plus a small unit
// descriptor; warp M issues the MMAs into two TMEM accumulators; 4*EW epilogue
// warps drain them reading only TMEM and the stage, and release the stage with
// the MMA. Units are split contiguously over a persistent grid, key-tile major
// so that consecutive units of a multi-query request reuse the same key tile.
#include <cstdint>
#include "kernels.cuh"

namespace dsa {


template <bool kFp8, int kHp, int kQG>
struct IndexerCfg {
  static constexpr int kAtoms = kFp8 ? 1 : 2;                  // 128-byte column blocks per row
  static constexpr int kN = kQG * kHp;                         // MMA N
  static constexpr int kKeyBytes = 128 * 128 * kAtoms;         // one 128-key tile
  static constexpr int kQBytes = kN * 128 * kAtoms;
  // per-stage side data: key scales (2 pages x 64), w and q_scale rows, unit descriptor
  static constexpr int kKsOff = kKeyBytes + kQBytes;
  static constexpr int kWOff = kKsOff + 512;
  static constexpr int kQsOff = kWOff + kN * 4;
  static constexpr int kDescOff = kQsOff + kN * 4;
  static constexpr int kSideBytes = ((512 + 2 * kN * 4 + 64) + 1023) / 1024 * 1024;
  static constexpr int kStageBytes = kKeyBytes + kQBytes + kSideBytes;
  static constexpr int kStages = (204800 / kStageBytes) < 8 ? (204800 / kStageBytes) : 8;
  static constexpr int kEW = kQG >= 2 ? 2 : 1;                 // epilogue warp groups
  static constexpr int kEpiWarps = 4 * kEW;
  static constexpr int kThreads = 32 * (kEpiWarps + 2);
  static constexpr int kProdWarp = kEpiWarps, kMmaWarp = kEpiWarps + 1;
  static constexpr int kTmemCols = (2 * kN) <= 32 ? 32 : (2 * kN) <= 64 ? 64 : (2 * kN) <= 128 ? 128
                                   : (2 * kN) <= 256 ? 256 : 512;
  static constexpr int kMaxB = 2048;                           // requests per call
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes;
  static constexpr int kKSteps = kFp8 ? 4 : 8;
  static_assert(kN <= 256 && kN % 16 == 0, "MMA N");
  static_assert(kStages >= 2, "stages");
};

// What the epilogue needs about a unit; written by the producer into the stage.
struct UnitDesc {
  int b, tile, q_start, q_count, len, pos0, page_ok;   // pos0 = position of the unit's first query
  int pad;
};

struct UnitInfo {
  int b, tile, q_start, q_count, len, q0, pos0;  // pos0 = position of the request's first query
};

template <int kQG>
__device__ __forceinline__ UnitInfo decode_unit(const int* prefix, int B, int u, const GeomDev& g) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {  // last b with prefix[b] <= u
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
  }
  UnitInfo ui;
  ui.b = lo;
  const int q0 = __ldg(g.cu_q + lo), q1 = __ldg(g.cu_q + lo + 1);
  const int nq = q1 - q0;
  const int ngroups = (nq + kQG - 1) / kQG;
  const int local = u - prefix[lo];
  ui.tile = local / ngroups;
  const int grp = local - ui.tile * ngroups;
  ui.q_start = q0 + grp * kQG;
  ui.q_count = min(kQG, nq - grp * kQG);
  ui.len = __ldg(g.seq_lens + lo);
  ui.q0 = q0;
  ui.pos0 = ui.len - nq;
  return ui;
}

template <bool kFp8, int kHp, int kQG>
__global__ void __launch_bounds__(IndexerCfg<kFp8, kHp, kQG>::kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_q,
                   const IndexerArgs A) {
  using C = IndexerCfg<kFp8, kHp, kQG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full_bar[C::kStages], empty_bar[C::kStages];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  __shared__ int prefix[C::kMaxB + 1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GeomDev& g = A.g;
  const int B = g.B;

  // ---- per-CTA unit table: prefix[b] = units before request b
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < B; base += 32) {
      const int b = base + lane;
      int units = 0;
      if (b < B) {
        const int q0 = __ldg(g.cu_q + b), q1 = __ldg(g.cu_q + b + 1), len = __ldg(g.seq_lens + b);
        const int nq = q1 - q0;
        const bool ok = nq >= 0 && nq <= len && len <= g.max_seq_len && q1 <= g.T;
        if (!ok) record_error(A.err, kDevBadIndex);
        else units = ((nq + kQG - 1) / kQG) * ((len + 127) / 128);
      }
      int incl = units;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (b < B) prefix[b] = run + incl - units;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[B] = run;
  }
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1 + C::kEpiWarps);   // MMA commit + every epilogue warp
    }
    for (int a = 0; a < 2; ++a) { mbar_init(smem_u32(&tfull_bar[a]), 1); mbar_init(smem_u32(&tempty_bar[a]), C::kEpiWarps); }
    fence_mbar_init();
  }
  // Query rows beyond Hi and w / q_scale entries beyond Hi stay zero for the whole
  // kernel (TMA and the bulk copies write only the first Hi of them).
  for (int s = 0; s < C::kStages; ++s) {
    int4* z = reinterpret_cast<int4*>(smem + s * C::kStageBytes + C::kKeyBytes);
    for (int i = tid; i < (C::kQBytes + C::kSideBytes) / 16; i += C::kThreads) z[i] = make_int4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (warp == C::kMmaWarp) { tmem_alloc(smem_u32(&tmem_base_s), C::kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  // The top-k grid that follows may start launching (it waits for these scores).
  griddep_launch_dependents();
  griddep_wait();   // a no-op unless this grid itself was launched programmatically

  const int U = prefix[B];
  const int G = gridDim.x;
  const int u_begin = (int)split_begin(blockIdx.x, U, G), u_end = (int)split_begin(blockIdx.x + 1, U, G);
  const int Hi = A.Hi;

  if (warp == C::kProdWarp) {
    // ================================================================ producer
    // 32 units are decoded at a time, one per lane, so their global lookups
    // overlap; lane 0 then fills one stage per unit.
    if (lane == 0) { tma_prefetch_desc(&map_k); tma_prefetch_desc(&map_q); }
    bool stop = false;
    for (int u_base = u_begin; u_base < u_end && !stop; u_base += 32) {
      const int u = u_base + lane;
      UnitInfo ui{};
      int pg0 = -1, pg1 = -1;
      if (u < u_end) {
        ui = decode_unit<kQG>(prefix, B, u, g);
        const int s0 = ui.tile * 128;
        const int* bt = g.block_table + (int64_t)ui.b * g.bt_stride;
        if (s0 < ui.len) pg0 = __ldg(bt + (s0 >> 6));
        if (s0 + 64 < ui.len) pg1 = __ldg(bt + ((s0 + 64) >> 6));
        const bool bad0 = s0 < ui.len && (pg0 < 0 || pg0 >= g.num_pages);
        const bool bad1 = s0 + 64 < ui.len && (pg1 < 0 || pg1 >= g.num_pages);
        if (bad0 || bad1) record_error(A.err, kDevBadIndex);
        if (bad0) pg0 = -1;
        if (bad1) pg1 = -1;
      }
      const int cnt = min(32, u_end - u_base);
      for (int jj = 0; jj < cnt; ++jj) {
        const int b = __shfl_sync(0xffffffffu, ui.b, jj), tile = __shfl_sync(0xffffffffu, ui.tile, jj);
        const int q_start = __shfl_sync(0xffffffffu, ui.q_start, jj), q_count = __shfl_sync(0xffffffffu, ui.q_count, jj);
        const int len = __shfl_sync(0xffffffffu, ui.len, jj);
        const int pos0 = __shfl_sync(0xffffffffu, ui.pos0 + (ui.q_start - ui.q0), jj);
        const int p0 = __shfl_sync(0xffffffffu, pg0, jj), p1 = __shfl_sync(0xffffffffu, pg1, jj);
        const int i = u_base + jj - u_begin;
        const int s = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        if (lane == 0) {
          if (!mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1, &abort_flag, A.err)) {
            stop = true;
          } else {
            uint8_t* st = smem + s * C::kStageBytes;
            UnitDesc* d = reinterpret_cast<UnitDesc*>(st + C::kDescOff);
            d->b = b; d->tile = tile; d->q_start = q_start; d->q_count = q_count; d->len = len; d->pos0 = pos0;
            d->page_ok = (p0 >= 0 ? 1 : 0) | (p1 >= 0 ? 2 : 0);
            const int np = (p0 >= 0) + (p1 >= 0);
            uint32_t bytes = np * 64 * 128 * C::kAtoms + q_count * Hi * 128 * C::kAtoms + q_count * Hi * 4;
            if (kFp8) bytes += np * 256 + q_count * Hi * 4;
            const uint32_t bar = smem_u32(&full_bar[s]);
            mbar_arrive_expect_tx(bar, bytes);
            const int pages[2] = {p0, p1};
            for (int hp = 0; hp < 2; ++hp) {
              if (pages[hp] < 0) continue;
              for (int a = 0; a < C::kAtoms; ++a)
                tma_load_2d(smem_u32(st + a * 16384 + hp * 8192), &map_k, bar, a * (kFp8 ? 128 : 64), pages[hp] * 64);
              if (kFp8) bulk_load(smem_u32(st + C::kKsOff + hp * 256), A.k_scale + (int64_t)pages[hp] * 64, 256, bar);
            }
            for (int j = 0; j < q_count; ++j) {
              const int t = q_start + j;
              for (int a = 0; a < C::kAtoms; ++a)
                tma_load_2d(smem_u32(st + C::kKeyBytes + a * (C::kN * 128) + j * kHp * 128), &map_q, bar,
                            a * (kFp8 ? 128 : 64), t * Hi);
              bulk_load(smem_u32(st + C::kWOff + j * kHp * 4), A.w + (int64_t)t * Hi, Hi * 4, bar);
              if (kFp8) bulk_load(smem_u32(st + C::kQsOff + j * kHp * 4), A.q_scale + (int64_t)t * Hi, Hi * 4, bar);
            }
          }
        }
        stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
        if (stop) break;
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(128, C::kN, kFp8 ? kFmtE4M3 : kFmtBF16, kFp8 ? kFmtE4M3 : kFmtBF16, 0, 0);
      for (int u = u_begin, i = 0; u < u_end; ++u, ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        const int acc = i & 1;
        const uint32_t aph = (i >> 1) & 1;
        if (!mbar_wait(smem_u32(&full_bar[s]), ph, &abort_flag, A.err)) break;
        if (!mbar_wait(smem_u32(&tempty_bar[acc]), aph ^ 1, &abort_flag, A.err)) break;
        tc_fence_after();
        const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
        const uint32_t qbase = kbase + C::kKeyBytes;
        const uint32_t d = tmem + acc * C::kN;
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk) {
          const uint32_t atom = kk / 4, within = (kk % 4) * 32;
          const uint64_t ad = smem_desc(kbase + atom * 16384 + within, 0, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(qbase + atom * (C::kN * 128) + within, 0, 1024, kSwizzle128B);
          if (kFp8) mma_f8_ss(d, ad, bd, idesc, kk > 0);
          else mma_f16_ss(d, ad, bd, idesc, kk > 0);
        }
        mma_commit(smem_u32(&empty_bar[s]));
        mma_commit(smem_u32(&tfull_bar[acc]));
      }
    }
  } else {
    // ================================================================ epilogue warps
    // Lane = key of the tile; reads the accumulator, the key scale, w and q_scale
    // from TMEM / the stage only.
    const int quarter = warp & 3, half = warp >> 2;
    const int key = quarter * 32 + lane;
    const float neg_inf = -__int_as_float(0x7f800000);
    for (int u = u_begin, i = 0; u < u_end; ++u, ++i) {
      const int s = i % C::kStages;
      const uint32_t ph = (i / C::kStages) & 1;
      const int acc = i & 1;
      const uint32_t aph = (i >> 1) & 1;
      if (!mbar_wait(smem_u32(&tfull_bar[acc]), aph, &abort_flag, A.err)) break;
      if (!mbar_wait(smem_u32(&full_bar[s]), ph, &abort_flag, A.err)) break;   // stage data visible here
      tc_fence_after();
      const uint8_t* st = smem + s * C::kStageBytes;
      const UnitDesc d = *reinterpret_cast<const UnitDesc*>(st + C::kDescOff);
      const float* wv = reinterpret_cast<const float*>(st + C::kWOff);
      const float* qv = reinterpret_cast<const float*>(st + C::kQsOff);
      const int sidx = d.tile * 128 + key;
      const bool in_ctx = sidx < d.len;
      const bool page_ok = (d.page_ok >> (key >> 6)) & 1;
      const float ks = kFp8 ? reinterpret_cast<const float*>(st + C::kKsOff)[key] : 1.f;
#pragma unroll 1
      for (int j = half; j < kQG; j += C::kEW) {
        if (j >= d.q_count) break;
        float sum = 0.f;
#pragma unroll
        for (int hc = 0; hc < kHp / 16; ++hc) {
          float v[16];
          tmem_ld16(tmem + acc * C::kN + j * kHp + hc * 16 + ((uint32_t)(quarter * 32) << 16), v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(wv + j * kHp + hc * 16 + e);
            if (kFp8) {
              const float4 q4 = *reinterpret_cast<const float4*>(qv + j * kHp + hc * 16 + e);
              sum = fmaf(w4.x * q4.x, fmaxf(v[e], 0.f), sum);
              sum = fmaf(w4.y * q4.y, fmaxf(v[e + 1], 0.f), sum);
              sum = fmaf(w4.z * q4.z, fmaxf(v[e + 2], 0.f), sum);
              sum = fmaf(w4.w * q4.w, fmaxf(v[e + 3], 0.f), sum);
            } else {
              sum = fmaf(w4.x, fmaxf(v[e], 0.f), sum);
              sum = fmaf(w4.y, fmaxf(v[e + 1], 0.f), sum);
              sum = fmaf(w4.z, fmaxf(v[e + 2], 0.f), sum);
              sum = fmaf(w4.w, fmaxf(v[e + 3], 0.f), sum);
            }
          }
        }
        if (in_ctx) {
          const int t = d.q_start + j;
          const int pos = d.pos0 + j;
          const float out = (sidx <= pos && page_ok) ? sum * ks : neg_inf;
          A.scores[(int64_t)t * A.stride + sidx] = out;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&tempty_bar[acc]));
        mbar_arrive(smem_u32(&empty_bar[s]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
template <bool kFp8, int kHp, int kQG>
static cudaError_t launch_indexer_t(const CUtensorMap& mk, const CUtensorMap& mq, const IndexerArgs& A,
                                    int grid, cudaStream_t st) {
  using C = IndexerCfg<kFp8, kHp, kQG>;
  auto kern = indexer_kernel<kFp8, kHp, kQG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(mk, mq, A);
  return cudaGetLastError();
}

int indexer_max_requests() { return IndexerCfg<true, 64, 1>::kMaxB; }

cudaError_t indexer_launch(bool fp8, int Hi, bool multi_query, const CUtensorMap& mk, const CUtensorMap& mq,
                           const IndexerArgs& A, int grid, cudaStream_t st) {
  const bool small = Hi <= 16;
  if (fp8) {
    if (small) return multi_query ? launch_indexer_t<true, 16, 4>(mk, mq, A, grid, st) : launch_indexer_t<true, 16, 1>(mk, mq, A, grid, st);
    return multi_query ? launch_indexer_t<true, 64, 4>(mk, mq, A, grid, st) : launch_indexer_t<true, 64, 1>(mk, mq, A, grid, st);
  }
  if (small) return multi_query ? launch_indexer_t<false, 16, 4>(mk, mq, A, grid, st) : launch_indexer_t<false, 16, 1>(mk, mq, A, grid, st);
  return multi_query ? launch_indexer_t<false, 64, 4>(mk, mq, A, grid, st) : launch_indexer_t<false, 64, 1>(mk, mq, A, grid, st);
}

}  // namespace dsa
