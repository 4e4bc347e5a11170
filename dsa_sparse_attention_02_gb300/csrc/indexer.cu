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
// one score per query, -inf past the query's causal position. The histogram variant
// (dsa_decode_step_hist) also counts the top 11 bits of each visible score's radix key
// per query and 16384-position chunk: the first pass of the radix top-k (lmdeploy
// "feat: support GLM-5.2", Changes) moved into the epilogue that makes the scores.
//
// Roles: warp P decodes 32 units at a time (one per lane) and, per unit, loads
// only what changed since the previous unit: a new key tile (two pages by TMA) into
// a ring of key stages, and a new query group
// (the QG x Hp query rows by TMA, w and q_scale by bulk copy) into a ring of query
// slots; a small descriptor per unit names the stage and slot it uses. A request's
// units run group-major: a query group is loaded once for all its key tiles (in
// decode the group is the request's one query; in prefill the 16 KB key tiles
// stream past the 32 KB group), and a group's QG consecutive queries arrive in one
// copy per operand. Warp M issues the MMAs into a ring of up to four TMEM
// accumulators; 4*EW epilogue warps drain them (one 64-column TMEM load per query;
// EW = 4 in the multi-query variant, one query per warp). The epilogue takes what it
// needs from a key stage (the key scales) and from a query slot (w * q_scale) when it
// first meets it and releases it at once, so a stage is held only until its MMAs
// complete. Units are split contiguously over a persistent grid.
#include <cstdint>
#include "kernels.cuh"

namespace dsa {


// Epilogue warp groups of the multi-query variant: four, so that each of the 16
// epilogue warps takes one query of a unit (more warps to hide the accumulator reads).
constexpr int kMultiEpiGroups = 4;

// kHistT: the first-digit histogram variant (its counters take dynamic shared memory).
template <bool kFp8, int kHp, int kQG, bool kHistT = false>
struct IndexerCfg {
  static constexpr int kAtoms = kFp8 ? 1 : 2;                  // 128-byte column blocks per row
  static constexpr int kN = kQG * kHp;                         // MMA N
  static constexpr int kKeyBytes = 128 * 128 * kAtoms;         // one 128-key tile
  // One-query units keep their tile's key scales in the key stage (copied with the
  // codes; the epilogue reads them there and releases the stage); query-group units
  // load them from global memory in the epilogue, so a stage holds codes alone and is
  // released by the MMA's commit (a fourth stage fits, and a handshake per unit goes).
  static constexpr bool kScaleInStage = kQG == 1;
  static constexpr int kKStageBytes = kKeyBytes + (kScaleInStage ? 1024 : 0);   // + key scales of its two pages (512 B)
  static constexpr int kQBytes = kN * 128 * kAtoms;            // the group's query rows
  static constexpr int kWOff = kQBytes, kQsOff = kQBytes + kN * 4;
  static constexpr int kQSlotBytes = (kQBytes + 2 * kN * 4 + 1023) / 1024 * 1024;
  static constexpr int kQSlots = (kQG >= 2 && kFp8) ? 4 : 2;
  // One-query e4m3 units run two CTAs per SM (two producers per SM), each with
  // half the shared memory; the other variants one CTA with the whole budget.
  static constexpr int kCtasPerSm = (kQG == 1 && kFp8) ? 2 : 1;
  // First-digit histograms (16-bit counts, two bins per word), in dynamic shared memory
  // after the key stages in the histogram variant: e4m3 keys only (the bf16
  // query-group variants have no room beside their operands; for bf16 keys the fused
  // step lets the top-k count the digit).
  static constexpr bool kHist = kFp8;
  static constexpr int kHistWords = kQG * kHistBins / 2;
  static constexpr int kHistBytes = kHist ? 4 * kHistWords + 16 : 0;   // + the two flush barriers
  // Dynamic shared memory for the operands: one CTA per SM keeps what it takes within
  // the 227 KB a CTA may hold beside at most 18 KB of static arrays and the histograms.
  static constexpr int kBudget1 = 232448 - 18432 - 1024 - (kHistT ? kHistBytes : 0);
  static constexpr int kBudget = kCtasPerSm == 2 ? 90112 : (kBudget1 < 204800 ? kBudget1 : 204800);
  static constexpr int kKStagesFit = (kBudget - kQSlots * kQSlotBytes) / kKStageBytes;
  static constexpr int kKStages = kKStagesFit < 8 ? kKStagesFit : 8;
  static constexpr int kDescs = 16;                            // unit descriptor ring
  static constexpr int kEW = kQG >= 2 ? kMultiEpiGroups : 1;   // epilogue warp groups
  static constexpr int kQPerWarp = kQG / kEW;                  // queries of a unit per epilogue warp
  static constexpr int kEpiWarps = 4 * kEW;
  static constexpr int kProdWarps = 1;
  static constexpr int kThreads = 32 * (kEpiWarps + kProdWarps + 1);
  // Register bound: warps are spread over the four SM sub-partitions, each with a
  // quarter of the register file, so the cap is set by the busiest one.
  static constexpr int kBoundThreads = 128 * ((kEpiWarps + kProdWarps + 1 + 3) / 4);
  // registers: kCtasPerSm CTAs of kBoundThreads share the register file
  static constexpr int kBoundCtas = kCtasPerSm;
  static constexpr int kProdWarp = kEpiWarps, kMmaWarp = kEpiWarps + kProdWarps;
  // TMEM accumulators: up to four, within this CTA's share of the 512 columns, so
  // that the MMA can run several units ahead of the epilogue.
  static constexpr int kAccsFit = (512 / kCtasPerSm) / kN;
  static constexpr int kAccs = kAccsFit >= 4 ? 4 : kAccsFit;
  static constexpr int kTmemCols = (kAccs * kN) <= 32 ? 32 : (kAccs * kN) <= 64 ? 64 : (kAccs * kN) <= 128 ? 128
                                   : (kAccs * kN) <= 256 ? 256 : 512;
  static constexpr int kMaxB = 1024;                           // requests per call
  static constexpr int kSmemBytes = 1024 + kQSlots * kQSlotBytes + kKStages * kKStageBytes;
  static constexpr int kKSteps = kFp8 ? 4 : 8;
  static_assert(kN <= 256 && kN % 16 == 0, "MMA N");
  static_assert(kKStages >= 2, "key stages");
  static_assert(kAccs >= 2 && kAccs * kN <= 512 / kCtasPerSm, "TMEM accumulators");
};

// What the MMA and epilogue warps need about a unit; written by the producer.
struct UnitDesc {
  int b, tile, q_start, q_count, len, pos0;   // pos0 = position of the unit's first query
  int page0, page1;                            // physical pages of the tile, -1 if unmapped
  int kstage, qslot;                           // key stage and query slot the unit reads
  int flags;                                   // bit 0: new key stage, bit 1: new query slot
};
constexpr int kNewKey = 1, kNewQuery = 2;

struct UnitInfo {
  int b, tile, q_start, q_count, len, q0, pos0;  // pos0 = position of the request's first query
};

template <int kQG>
// prefix, cuq and lens are shared-memory copies of the unit prefix, cu_q and seq_lens.
__device__ __forceinline__ UnitInfo decode_unit(const int* prefix, const int* cuq, const int* lens, int B, int tile0,
                                                int u) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {  // last b with prefix[b] <= u
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
  }
  UnitInfo ui;
  ui.b = lo;
  const int q0 = cuq[lo], q1 = cuq[lo + 1];
  const int nq = q1 - q0;
  const int ngroups = (nq + kQG - 1) / kQG;
  // group-major: a unit run keeps its query group and streams the key tiles (a
  // group's queries are loaded once; tiles are the smaller operand)
  const int ntiles = (prefix[lo + 1] - prefix[lo]) / ngroups;
  const int local = u - prefix[lo];
  const int grp = local / ntiles;
  const int lt = local - grp * ntiles;
  ui.tile = tile0 + lt;
  ui.q_start = q0 + grp * kQG;
  ui.q_count = min(kQG, nq - grp * kQG);
  ui.len = lens[lo];
  ui.q0 = q0;
  ui.pos0 = ui.len - nq;
  return ui;
}

// Adds the shared first-digit histograms of queries hq .. hq+hn-1 (chunk hc) into the
// global ones and clears them; every epilogue warp calls it at the same point of the
// unit sequence (the barriers' phase hph), each taking its share of the words.
template <int kEpiWarps>
__device__ __noinline__ bool hist_flush(uint32_t* hist_s, int hq, int hc, int hn, uint32_t& hph, uint32_t full,
                                        uint32_t empty, const IndexerArgs& A, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (lane == 0) mbar_arrive(full);          // this warp's counts are in
  if (!mbar_wait(full, hph & 1, abort_flag, A.err)) return false;
  for (int i = threadIdx.x; i < hn * (kHistBins / 2); i += 32 * kEpiWarps) {
    const uint32_t v = hist_s[i];
    if (v != 0u) {
      const int j = i / (kHistBins / 2), bin = 2 * (i % (kHistBins / 2));
      int* dst = A.hist + ((int64_t)(hq + j) * A.hist_chunks + hc) * kHistBins + bin;
      if (v & 0xffffu) atomicAdd(dst, (int)(v & 0xffffu));
      if (v >> 16) atomicAdd(dst + 1, (int)(v >> 16));
      hist_s[i] = 0u;
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty);         // this warp's share is cleared
  if (!mbar_wait(empty, hph & 1, abort_flag, A.err)) return false;
  ++hph;
  return true;
}

// kHistT: the variant that also counts first-digit histograms (A.hist set).
template <bool kFp8, int kHp, int kQG, bool kHistT>
__global__ void __launch_bounds__(IndexerCfg<kFp8, kHp, kQG>::kBoundThreads, IndexerCfg<kFp8, kHp, kQG>::kBoundCtas)
    indexer_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_q,
                   const IndexerArgs A) {
  using C = IndexerCfg<kFp8, kHp, kQG, kHistT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_slots = smem;                                       // kQSlots x kQSlotBytes
  uint8_t* k_stages = smem + C::kQSlots * C::kQSlotBytes;        // kKStages x kKStageBytes
  __shared__ uint64_t key_full[C::kKStages], key_empty[C::kKStages];
  __shared__ uint64_t q_full[C::kQSlots], q_empty[C::kQSlots];
  __shared__ uint64_t desc_full[C::kDescs], desc_empty[C::kDescs];
  __shared__ uint64_t tfull_bar[C::kAccs], tempty_bar[C::kAccs];
  // w * q_scale of the current query group, one copy per epilogue warp
  constexpr bool kWqRegs = kQG == 1 && C::kCtasPerSm == 1;
  __shared__ __align__(16) float wq_s[kWqRegs ? 1 : C::kEpiWarps][kWqRegs ? 4 : C::kQPerWarp * kHp];
  __shared__ UnitDesc descs[C::kDescs];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  // First-digit histograms of the query group being scored (A.hist set: the launch's
  // dynamic shared memory holds them after the key stages): 16-bit counts, two bins per
  // word (a group's count in one bin and chunk is at most 16384), added to the global
  // histograms when the group or the 16384-position chunk changes and at the end, the
  // epilogue warps meeting on two barriers after them around it.
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(k_stages + C::kKStages * C::kKStageBytes);
  uint64_t* hist_bars = reinterpret_cast<uint64_t*>(hist_s + C::kHistWords);   // full, empty
  __shared__ int prefix[C::kMaxB + 1], cuq_s[C::kMaxB + 1], lens_s[C::kMaxB];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GeomDev& g = A.g;
  const int B = g.B;

  // ---- per-CTA unit table: prefix[b] = units before request b. The request
  // metadata is read in one round trip by every thread; meanwhile the CTAs warm the
  // block table in L2 (a slice each), which the producer reads next.
  {
    const int64_t bt_lines = ((int64_t)B * g.bt_stride * 4 + 127) / 128;
    if (tid >= 32 && tid < 64)
      for (int64_t l = blockIdx.x + (int64_t)gridDim.x * (tid - 32); l < bt_lines; l += (int64_t)gridDim.x * 32)
        prefetch_l2(reinterpret_cast<const uint8_t*>(g.block_table) + l * 128);
    for (int b = tid; b <= B; b += C::kThreads) {
      cuq_s[b] = __ldg(g.cu_q + b);
      if (b < B) lens_s[b] = __ldg(g.seq_lens + b);
    }
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < B; base += 32) {
      const int b = base + lane;
      int units = 0;
      if (b < B) {
        const int q0 = cuq_s[b], q1 = cuq_s[b + 1], len = lens_s[b];
        const int nq = q1 - q0;
        const bool ok = nq >= 0 && nq <= len && len <= g.max_seq_len && q1 <= g.T;
        if (!ok) record_error(A.err, kDevBadIndex);
        else units = ((nq + kQG - 1) / kQG) * max(0, (min(len, A.key_end) + 127) / 128 - A.key_begin / 128);
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
    // a stage / slot is released by the MMA thread's commit and every epilogue
    // warp once they have moved on to the next one
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(smem_u32(&key_full[s]), 1);
      mbar_init(smem_u32(&key_empty[s]), 1 + (C::kScaleInStage ? C::kEpiWarps : 0));
    }
    for (int s = 0; s < C::kQSlots; ++s) { mbar_init(smem_u32(&q_full[s]), 1); mbar_init(smem_u32(&q_empty[s]), 1 + C::kEpiWarps); }
    for (int s = 0; s < C::kDescs; ++s) { mbar_init(smem_u32(&desc_full[s]), 1); mbar_init(smem_u32(&desc_empty[s]), 1 + C::kEpiWarps); }
    for (int a = 0; a < C::kAccs; ++a) { mbar_init(smem_u32(&tfull_bar[a]), 1); mbar_init(smem_u32(&tempty_bar[a]), C::kEpiWarps); }
    if constexpr (kHistT) {
      mbar_init(smem_u32(&hist_bars[0]), C::kEpiWarps);
      mbar_init(smem_u32(&hist_bars[1]), C::kEpiWarps);
    }
    fence_mbar_init();
  }
  if constexpr (kHistT)
    for (int i = tid; i < C::kHistWords; i += C::kThreads) hist_s[i] = 0u;
  // Query rows beyond Hi and w / q_scale entries beyond Hi stay zero for the whole
  // kernel (TMA and the bulk copies write only the first Hi of them).
  for (int i = tid; i < C::kQSlots * C::kQSlotBytes / 16; i += C::kThreads)
    reinterpret_cast<int4*>(q_slots)[i] = make_int4(0, 0, 0, 0);
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
    // overlap; lane 0 then publishes one descriptor per unit, loading a key tile
    // or a query group only when it differs from the previous unit's.
    if (lane == 0) { tma_prefetch_desc(&map_k); tma_prefetch_desc(&map_q); }
    bool stop = false;
    int kcount = 0, qcount = 0;                       // key stages / query slots opened so far
    int prev_b = -1, prev_tile = -1, prev_q = -1;
    for (int u_base = u_begin; u_base < u_end && !stop; u_base += 32) {
      const int u = u_base + lane;
      UnitInfo ui{};
      int pg0 = -1, pg1 = -1;
      if (u < u_end) {
        ui = decode_unit<kQG>(prefix, cuq_s, lens_s, B, A.key_begin / 128, u);
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
        if (lane == 0) {
          const int r = i % C::kDescs;
          const bool new_k = (b != prev_b) || (tile != prev_tile);
          const bool new_q = (b != prev_b) || (q_start != prev_q);
          // a descriptor slot is fresh on the ring's first lap
          bool ok = i < C::kDescs || mbar_wait(smem_u32(&desc_empty[r]), ((i / C::kDescs) & 1) ^ 1, &abort_flag, A.err);
          if (ok && new_k) {
            const int ks = kcount % C::kKStages;
            ok = mbar_wait(smem_u32(&key_empty[ks]), ((kcount / C::kKStages) & 1) ^ 1, &abort_flag, A.err);
            if (ok) {
              uint8_t* st = k_stages + ks * C::kKStageBytes;
              const uint32_t bar = smem_u32(&key_full[ks]);
              const int np = (p0 >= 0) + (p1 >= 0);
              mbar_arrive_expect_tx(bar, np * 64 * 128 * C::kAtoms + (kFp8 && C::kScaleInStage ? np * 256 : 0));
              const int pages[2] = {p0, p1};
              for (int hp = 0; hp < 2; ++hp) {
                if (pages[hp] < 0) continue;
                for (int a = 0; a < C::kAtoms; ++a)
                  tma_load_2d(smem_u32(st + a * 16384 + hp * 8192), &map_k, bar, a * (kFp8 ? 128 : 64), pages[hp] * 64);
                if (kFp8 && C::kScaleInStage)
                  bulk_load(smem_u32(st + C::kKeyBytes + hp * 256), A.k_scale + (int64_t)pages[hp] * 64, 256, bar);
              }
              ++kcount;
            }
          }
          if (ok && new_q) {
            const int qs = qcount % C::kQSlots;
            ok = mbar_wait(smem_u32(&q_empty[qs]), ((qcount / C::kQSlots) & 1) ^ 1, &abort_flag, A.err);
            if (ok) {
              uint8_t* sl = q_slots + qs * C::kQSlotBytes;
              const uint32_t bar = smem_u32(&q_full[qs]);
              // w and q_scale rows of Hi floats are bulk-copied when Hi * 4 is a multiple
              // of 16 bytes; otherwise they go as 4-byte copies whose completion the barrier
              // also tracks (that arrival is registered before the expect_tx arrival, so the
              // phase cannot complete without them).
              const bool vec = (Hi & 3) == 0;
              if (!vec) {
                for (int j = 0; j < q_count; ++j) {
                  const int64_t t = q_start + j;
                  for (int h = 0; h < Hi; ++h) {
                    cp_async_4(smem_u32(sl + C::kWOff + (j * kHp + h) * 4), A.w + t * Hi + h, 4u);
                    if (kFp8) cp_async_4(smem_u32(sl + C::kQsOff + (j * kHp + h) * 4), A.q_scale + t * Hi + h, 4u);
                  }
                }
                cp_async_arrive(bar);
              }
              if (kQG > 1 && A.q_group_box) {
                // the group's rows are consecutive in q, w and q_scale, and Hi == kHp lays
                // them out in the slot as one box: one copy per atom and per vector (a box
                // past the last query is zero-filled and counted in full)
                mbar_arrive_expect_tx(bar, kQG * Hi * 128 * C::kAtoms + q_count * Hi * (kFp8 ? 8 : 4));
                for (int a = 0; a < C::kAtoms; ++a)
                  tma_load_2d(smem_u32(sl + a * (C::kN * 128)), &map_q, bar, a * (kFp8 ? 128 : 64), q_start * Hi);
                bulk_load(smem_u32(sl + C::kWOff), A.w + (int64_t)q_start * Hi, q_count * Hi * 4, bar);
                if (kFp8) bulk_load(smem_u32(sl + C::kQsOff), A.q_scale + (int64_t)q_start * Hi, q_count * Hi * 4, bar);
              } else {
              mbar_arrive_expect_tx(bar, q_count * Hi * (128 * C::kAtoms + (vec ? 4 + (kFp8 ? 4 : 0) : 0)));
              for (int j = 0; j < q_count; ++j) {
                const int t = q_start + j;
                for (int a = 0; a < C::kAtoms; ++a)
                  tma_load_2d(smem_u32(sl + a * (C::kN * 128) + j * kHp * 128), &map_q, bar, a * (kFp8 ? 128 : 64), t * Hi);
                if (vec) {
                  bulk_load(smem_u32(sl + C::kWOff + j * kHp * 4), A.w + (int64_t)t * Hi, Hi * 4, bar);
                  if (kFp8) bulk_load(smem_u32(sl + C::kQsOff + j * kHp * 4), A.q_scale + (int64_t)t * Hi, Hi * 4, bar);
                }
              }
              }
              ++qcount;
            }
          }
          if (ok) {
            UnitDesc& d = descs[r];
            d.b = b; d.tile = tile; d.q_start = q_start; d.q_count = q_count; d.len = len; d.pos0 = pos0;
            d.page0 = p0; d.page1 = p1;
            d.kstage = (kcount - 1) % C::kKStages;
            d.qslot = (qcount - 1) % C::kQSlots;
            d.flags = (new_k ? kNewKey : 0) | (new_q ? kNewQuery : 0);
            mbar_arrive(smem_u32(&desc_full[r]));
            prev_b = b; prev_tile = tile; prev_q = q_start;
          }
          stop = !ok;
        }
        stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
        if (stop) break;
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(128, C::kN, kFp8 ? kFmtE4M3 : kFmtBF16, kFp8 ? kFmtE4M3 : kFmtBF16, 0, 0);
      int kc = 0, qc = 0, cur_k = -1, cur_q = -1;
      for (int u = u_begin, i = 0; u < u_end; ++u, ++i) {
        const int r = i % C::kDescs;
        if (!mbar_wait(smem_u32(&desc_full[r]), (i / C::kDescs) & 1, &abort_flag, A.err)) break;
        const UnitDesc d = descs[r];
        mbar_arrive(smem_u32(&desc_empty[r]));
        if (d.flags & kNewKey) {
          if (cur_k >= 0) mma_commit(smem_u32(&key_empty[cur_k]));   // after every MMA that read it
          cur_k = d.kstage;
          if (!mbar_wait(smem_u32(&key_full[cur_k]), (kc / C::kKStages) & 1, &abort_flag, A.err)) break;
          ++kc;
        }
        if (d.flags & kNewQuery) {
          if (cur_q >= 0) mma_commit(smem_u32(&q_empty[cur_q]));
          cur_q = d.qslot;
          if (!mbar_wait(smem_u32(&q_full[cur_q]), (qc / C::kQSlots) & 1, &abort_flag, A.err)) break;
          ++qc;
        }
        const int acc = i % C::kAccs;
        if (!mbar_wait(smem_u32(&tempty_bar[acc]), ((i / C::kAccs) & 1) ^ 1, &abort_flag, A.err)) break;
        tc_fence_after();
        const uint64_t a0 = smem_desc(smem_u32(k_stages + cur_k * C::kKStageBytes), 0, 1024, kSwizzle128B);
        const uint64_t b0 = smem_desc(smem_u32(q_slots + cur_q * C::kQSlotBytes), 0, 1024, kSwizzle128B);
        const uint32_t dt = tmem + acc * C::kN;
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk) {
          const uint32_t atom = kk / 4, within = (kk % 4) * 32;
          const uint64_t ad = desc_add(a0, atom * 16384 + within);
          const uint64_t bd = desc_add(b0, atom * (C::kN * 128) + within);
          if (kFp8) mma_f8_ss(dt, ad, bd, idesc, kk > 0);
          else mma_f16_ss(dt, ad, bd, idesc, kk > 0);
        }
        mma_commit(smem_u32(&tfull_bar[acc]));
      }
    }
  } else {
    // ================================================================ epilogue warps
    // Lane = key of the tile. The key's scale: read from a new key stage, which is then
    // released at once (one-query units; the MMA's commit covers its own reads), or
    // loaded from global memory when the unit starts (query groups). A new query
    // group: w * q_scale is formed once (registers for one query and one CTA per SM,
    // else this warp's shared copy) and the slot released. Then per unit only the
    // accumulator (TMEM) is read.
    const int quarter = warp & 3, half = warp >> 2;
    const int key = quarter * 32 + lane;
    const float neg_inf = -__int_as_float(0x7f800000);
    int kc = 0, qc = 0, cur_k = -1, cur_q = -1;
    float ks = 1.f;
    float wq[kWqRegs ? kHp : 1];
    const float* wqw = &wq_s[kWqRegs ? 0 : warp][0];
    // the shared histograms count queries hq .. hq+hn-1 in chunk hc (hq < 0: none yet)
    int hq = -1, hc = 0, hn = 0;
    uint32_t hph = 0;
    for (int u = u_begin, i = 0; u < u_end; ++u, ++i) {
      const int r = i % C::kDescs;
      if (!mbar_wait(smem_u32(&desc_full[r]), (i / C::kDescs) & 1, &abort_flag, A.err)) break;
      const UnitDesc d = descs[r];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&desc_empty[r]));
      if constexpr (kHistT) {
        const int chunk = d.tile >> (kTopkChunkLog2 - 7);   // 128-key tiles
        if (d.q_start != hq || chunk != hc) {
          if (hq >= 0 && !hist_flush<C::kEpiWarps>(hist_s, hq, hc, hn, hph, smem_u32(&hist_bars[0]),
                                                   smem_u32(&hist_bars[1]), A, &abort_flag))
            break;
          hq = d.q_start; hc = chunk; hn = d.q_count;
        }
      }
      const int page = (key < 64) ? d.page0 : d.page1;   // -1 if unmapped or out of range
      if constexpr (C::kScaleInStage) {
        if (d.flags & kNewKey) {
          cur_k = d.kstage;
          if (!mbar_wait(smem_u32(&key_full[cur_k]), (kc / C::kKStages) & 1, &abort_flag, A.err)) break;   // key scales visible
          ++kc;
          if (kFp8) ks = reinterpret_cast<const float*>(k_stages + cur_k * C::kKStageBytes + C::kKeyBytes)[key];
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&key_empty[cur_k]));
        }
      } else if (kFp8) {
        ks = page >= 0 ? __ldg(A.k_scale + (int64_t)page * 64 + (key & 63)) : 1.f;
      }
      if (d.flags & kNewQuery) {
        cur_q = d.qslot;
        if (!mbar_wait(smem_u32(&q_full[cur_q]), (qc / C::kQSlots) & 1, &abort_flag, A.err)) break;   // w, q_scale visible
        ++qc;
        const uint8_t* sl = q_slots + cur_q * C::kQSlotBytes;
        if constexpr (kWqRegs) {
#pragma unroll
          for (int e = 0; e < kHp; e += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(sl + C::kWOff + e * 4);
            float4 q4 = make_float4(1.f, 1.f, 1.f, 1.f);
            if (kFp8) q4 = *reinterpret_cast<const float4*>(sl + C::kQsOff + e * 4);
            wq[e] = w4.x * q4.x; wq[e + 1] = w4.y * q4.y; wq[e + 2] = w4.z * q4.z; wq[e + 3] = w4.w * q4.w;
          }
        } else {
          __syncwarp();   // the previous group's copy has been read by every lane
          const float* wv = reinterpret_cast<const float*>(sl + C::kWOff);
          const float* qv = reinterpret_cast<const float*>(sl + C::kQsOff);
          // this warp's queries of the group: half, half + kEW, ...
#pragma unroll
          for (int jj = 0; jj < C::kQPerWarp; ++jj) {
            const int o = (half + jj * C::kEW) * kHp;
            for (int e = lane; e < kHp; e += 32) wq_s[warp][jj * kHp + e] = wv[o + e] * (kFp8 ? qv[o + e] : 1.f);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&q_empty[cur_q]));
      }
      const int acc = i % C::kAccs;
      if (!mbar_wait(smem_u32(&tfull_bar[acc]), (i / C::kAccs) & 1, &abort_flag, A.err)) break;
      tc_fence_after();
      const int sidx = d.tile * 128 + key;
      const bool in_ctx = sidx < d.len && sidx < A.key_end;
#pragma unroll 1
      for (int jj = 0; jj < C::kQPerWarp; ++jj) {
        const int j = half + jj * C::kEW;
        if (j >= d.q_count) break;
        float v[kHp];
        if constexpr (kHp == 64) tmem_ld64(tmem + acc * C::kN + j * kHp + ((uint32_t)(quarter * 32) << 16), v);
        else tmem_ld16(tmem + acc * C::kN + j * kHp + ((uint32_t)(quarter * 32) << 16), v);
        tmem_ld_wait();
        // four partial sums (heads e, e+1, e+2, e+3 mod 4) as two packed pairs, added at
        // the end in the same order as four scalar sums would be
        float2 s2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int e = 0; e < kHp; e += 4) {
          float2 c0, c1;
          if constexpr (kWqRegs) {
            c0 = make_float2(wq[e], wq[e + 1]); c1 = make_float2(wq[e + 2], wq[e + 3]);
          } else {
            const float4 w4 = *reinterpret_cast<const float4*>(wqw + jj * kHp + e);
            c0 = make_float2(w4.x, w4.y); c1 = make_float2(w4.z, w4.w);
          }
          s2[0] = __ffma2_rn(c0, make_float2(fmaxf(v[e], 0.f), fmaxf(v[e + 1], 0.f)), s2[0]);
          s2[1] = __ffma2_rn(c1, make_float2(fmaxf(v[e + 2], 0.f), fmaxf(v[e + 3], 0.f)), s2[1]);
        }
        const float sum = (s2[0].x + s2[0].y) + (s2[1].x + s2[1].y);
        if (in_ctx) {
          const int t = d.q_start + j;
          const int pos = d.pos0 + j;
          const float out = (sidx <= pos && page >= 0) ? sum * ks : neg_inf;
          A.scores[(int64_t)t * A.stride + (sidx - A.key_begin)] = out;
          if constexpr (kHistT) {
            if (sidx <= pos) {
              // first-digit histogram of the positions the top-k selects from (0..pos)
              const uint32_t bin = orderable_key(out) >> kHistShift;
              atomicAdd(&hist_s[j * (kHistBins / 2) + (bin >> 1)], 1u << ((bin & 1u) << 4));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[acc]));
    }
    if constexpr (kHistT)
      if (hq >= 0) hist_flush<C::kEpiWarps>(hist_s, hq, hc, hn, hph, smem_u32(&hist_bars[0]), smem_u32(&hist_bars[1]),
                                            A, &abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// The geometry of queries [t0, t1) alone (bounded scoring, lmdeploy "glm5.3-flash
// support", Capacity improvement: bounded KPool scoring): request b keeps the part
// of its queries inside the range, and its length becomes the last such query's
// position + 1, so every kept query keeps its position (L - n + j) and the keys it
// can see; a request with no query in the range gets none and length 0.
__global__ void query_ranges_kernel(const int* __restrict__ cu_q, const int* __restrict__ seq_lens, int B, int T,
                                    int t_first, int rows, int* __restrict__ out, int stride) {
  // block j: the range of queries [t_first + j*rows, +rows) into out + j*stride (cu_q
  // of the range, then its lengths)
  const int t0 = t_first + blockIdx.x * rows, t1 = min(t0 + rows, T);
  int* cu_out = out + (int64_t)blockIdx.x * stride;
  int* len_out = cu_out + B + 1;
  for (int b = threadIdx.x; b <= B; b += blockDim.x) {
    const int q0 = cu_q[b];
    cu_out[b] = min(max(q0, t0), t1) - t0;
    if (b < B) {
      const int q1 = cu_q[b + 1];
      const int n = min(q1, t1) - max(q0, t0);
      len_out[b] = n > 0 ? seq_lens[b] - (q1 - min(q1, t1)) : 0;
    }
  }
}

cudaError_t query_ranges_launch(const int* cu_q, const int* seq_lens, int B, int T, int t_first, int rows, int n,
                                int* out, int stride, cudaStream_t st) {
  query_ranges_kernel<<<n, 1024, 0, st>>>(cu_q, seq_lens, B, T, t_first, rows, out, stride);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ host side
template <bool kFp8, int kHp, int kQG, bool kHistT = false>
static cudaError_t launch_indexer_t(const CUtensorMap& mk, const CUtensorMap& mq, const IndexerArgs& A,
                                    int grid, bool pdl, cudaStream_t st) {
  using C = IndexerCfg<kFp8, kHp, kQG, kHistT>;
  if constexpr (!kHistT) {
    if (A.hist != nullptr) {
      if constexpr (C::kHist) return launch_indexer_t<kFp8, kHp, kQG, true>(mk, mq, A, grid, pdl, st);
      return cudaErrorInvalidValue;   // indexer_counts_hist() said no
    }
  }
  auto kern = indexer_kernel<kFp8, kHp, kQG, kHistT>;
  const int smem = C::kSmemBytes + (kHistT ? C::kHistBytes : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid * C::kCtasPerSm, 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at; cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mk, mq, A);
}

int indexer_max_requests() { return IndexerCfg<true, 64, 1>::kMaxB; }

bool indexer_counts_hist(bool fp8, int, bool) { return fp8 && IndexerCfg<true, 64, 4>::kHist; }

int indexer_q_box_rows(int Hi, bool multi_query) {
  return multi_query && (Hi == 16 || Hi == 64) ? 4 * Hi : Hi;
}

cudaError_t indexer_launch(bool fp8, int Hi, bool multi_query, const CUtensorMap& mk, const CUtensorMap& mq,
                           const IndexerArgs& A, int grid, bool pdl, cudaStream_t st) {
  const bool small = Hi <= 16;
  if (fp8) {
    if (small) return multi_query ? launch_indexer_t<true, 16, 4>(mk, mq, A, grid, pdl, st) : launch_indexer_t<true, 16, 1>(mk, mq, A, grid, pdl, st);
    return multi_query ? launch_indexer_t<true, 64, 4>(mk, mq, A, grid, pdl, st) : launch_indexer_t<true, 64, 1>(mk, mq, A, grid, pdl, st);
  }
  if (small) return multi_query ? launch_indexer_t<false, 16, 4>(mk, mq, A, grid, pdl, st) : launch_indexer_t<false, 16, 1>(mk, mq, A, grid, pdl, st);
  return multi_query ? launch_indexer_t<false, 64, 4>(mk, mq, A, grid, pdl, st) : launch_indexer_t<false, 64, 1>(mk, mq, A, grid, pdl, st);
}

}  // namespace dsa
