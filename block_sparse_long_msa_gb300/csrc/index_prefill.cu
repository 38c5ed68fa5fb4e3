// Index branch for prefill, fused: raw index scores (tcgen05 GEMM) -> 128-token block max-pool
// -> per-group top-(k-1) of the earlier blocks -> + local block.  The L x L score matrix never
// leaves the SM: each score tile lives in TMEM only until its row maxima are taken.
//
// Method: "MiniMax M3 算力省 20 倍", section 二 (index scores over the causal window, max-pooling,
// per-group top-k, forced local block) and section 四 (exp-free top-k: ranking uses raw scores).
//
// One CTA owns one query block qb (128 queries) for gpc groups (two when G is even, else one).
// The gpc index-query tiles stay in shared memory; the keys of blocks 0..qb-1 stream through a
// TMA ring in tiles of 256 keys (two blocks), so every MMA is M=128 x N=256 (x K=16 in bf16,
// K=32 in e4m3): the tensor core runs an N=256 step in about the time of an N=128 one.  Score
// tiles go to two 256-column TMEM accumulators; work unit u = (key tile u / gpc, group u % gpc)
// takes slot u & 1, so with two groups each slot belongs to one group and each group's MMAs
// overlap the other group's epilogue.  Roles:
//   warps 0..7  two epilogue warpgroups; warpgroup e drains slot e: thread r owns query row r and
//               takes the two block maxima of its 256 scores straight from the TMEM loads
//               (tcgen05.ld.red), then keeps a register top-15
//   warp 8      TMA producer (index-query tiles once, then key tiles)
//   warp 9      TMEM owner + single-thread tcgen05.mma issuer, which polls its barriers
// A slot is MMA'd, then drained, then MMA'd again, so each slot's round trip (MMAs done, commit,
// drain, release, the next MMAs issued) must hide behind the other slot's MMAs; at the fp8 rate
// four MMA steps do not cover it.
// With one group per CTA the two warpgroups see alternate key tiles and merge their lists at the
// end; the full (score desc, block asc) comparison of the list keeps the tie rule.
#include "common.cuh"
#include "launch.h"

namespace msa {

namespace {

// Wait for the phase by polling (mbarrier.test_wait, never suspended); gives up after limit_ns
// of wall time, read every 256 polls.  Used by the single MMA-issuing thread: a suspended
// try_wait wakes up later than the phase completes, and that delay sits between one slot's MMAs
// and the next (L = 1M: 334.6 -> 322.9 ms in bf16, 255.3 -> 248.8 ms in e4m3).  The epilogue
// warps keep mbar_wait: polling there takes issue slots from their own work and was slower.
__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  uint64_t t0 = 0;
  uint32_t n = 0;
  while (!mbar_test_wait(bar, parity)) {
    if ((++n & 255u) == 0) {
      const uint64_t t = globaltimer_ns();
      if (t0 == 0)
        t0 = t;
      else if (t - t0 > limit_ns)
        return false;
    }
  }
  return true;
}

// Tiles of index vectors (128 elements), K-major with the 128-byte swizzle: a bf16 row is two
// 128-byte panels (64 elements each), an e4m3 row one.  Every MMA step covers 32 bytes of K
// (16 bf16 or 32 e4m3 elements), so K = 128 takes 8 bf16 steps or 4 e4m3 steps.
template <bool kF8>
struct IdxTiles {
  static constexpr uint32_t kEsz = kF8 ? 1 : 2;
  static constexpr uint32_t kQPanel = 128 * 128;                 // 128 rows x 128 bytes
  static constexpr uint32_t kQTile = 128 * kDim * kEsz;
  static constexpr uint32_t kKPanel = kIndexKeyTile * 128;
  static constexpr uint32_t kKTile = kIndexKeyTile * kDim * kEsz;
  static constexpr int kPanels = kF8 ? 1 : 2;
  static constexpr int kSteps = kF8 ? 4 : 8;
  static constexpr uint32_t kIdesc = kF8 ? idesc_e4m3_f32(128, kIndexKeyTile)
                                         : idesc_bf16_f32(128, kIndexKeyTile, false, false);
  static constexpr int kMaxStages = kF8 ? 6 : 3;
};
constexpr int kMaxStagesIdx = 6;
static_assert(kIndexKeyTile == 2 * kBlock, "a key tile is two blocks");

// barrier block (offsets from its start)
constexpr uint32_t kBarQ = 0;                              // index-query tiles landed
constexpr uint32_t kBarFull = 8;                           // [8, 8 + 8 * kMaxStagesIdx)
constexpr uint32_t kBarEmpty = kBarFull + 8 * kMaxStagesIdx;
constexpr uint32_t kBarAccFull = kBarEmpty + 8 * kMaxStagesIdx;  // two slots
constexpr uint32_t kBarAccEmpty = kBarAccFull + 16;
constexpr uint32_t kBarDrain = kBarAccEmpty + 16;
constexpr uint32_t kTmemSlotOff = kBarDrain + 8;
constexpr uint32_t kAbortOff = kTmemSlotOff + 4;
constexpr uint32_t kBarBytes = 256;
static_assert(kAbortOff + 4 <= kBarBytes, "barrier block");

struct IndexPrefillArgs {
  int64_t L;
  int32_t G, gpc, k, nb, ns;
  int32_t* sel;
  float* sel_score;
  float* block_scores;  // optional [G][L][nb]: every block's pooled score (+inf local, -inf later)
  int32_t* status;
  uint64_t wait_ns;
  // Key blocks scored: [kb0, kb1) (the whole causal range: 0, nb).  The key tensor map starts at
  // block kb0.  With cand_block set, each row's top-(k-1) of those blocks is written in rank
  // order to cand_score / cand_block [G][L][k-1] (a shard of the context-parallel index branch)
  // instead of the selection.
  int32_t kb0, kb1;
  float* cand_score;
  int32_t* cand_block;
};

// Shared memory: gpc index-query tiles, ns key stages, then the barrier block.
constexpr int kIndexThreads = 320;
constexpr int kWarpProducer = 8, kWarpMma = 9;

template <bool kF8>
__global__ void __launch_bounds__(kIndexThreads, 1)
    index_select_prefill_kernel(const __grid_constant__ CUtensorMap map_q,
                                const __grid_constant__ CUtensorMap map_k, IndexPrefillArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  using T = IdxTiles<kF8>;
  constexpr uint32_t kQTile = T::kQTile, kQPanel = T::kQPanel, kKTile = T::kKTile,
                     kKPanel = T::kKPanel;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int gpc = a.gpc, ns = a.ns;
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + gpc * kQTile;
  const uint32_t bars = sK + ns * kKTile;
  const uint32_t bar_q = bars + kBarQ;
  auto b_full = [&](int s) { return bars + kBarFull + 8 * s; };
  auto b_empty = [&](int s) { return bars + kBarEmpty + 8 * s; };
  auto acc_full = [&](int t) { return bars + kBarAccFull + 8 * t; };
  auto acc_empty = [&](int t) { return bars + kBarAccEmpty + 8 * t; };
  const uint32_t drain_bar = bars + kBarDrain;
  uint8_t* bar_ptr = smem + (bars - sQ);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_ptr + kTmemSlotOff);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(bar_ptr + kAbortOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cpq = a.G / gpc;                                    // CTAs per query block
  const int qb = a.nb - 1 - static_cast<int>(blockIdx.x) / cpq;  // heaviest query blocks first
  const int g0 = (static_cast<int>(blockIdx.x) % cpq) * gpc;
  // key blocks kb0 .. kb0+nkey-1: those of the range strictly before the query block
  const int nkey = max(0, min(a.kb1, qb) - a.kb0);
  const int ntiles = (nkey + 1) / 2;
  const int nunits = ntiles * gpc;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < ns; ++s) {
      mbar_init(b_full(s), 1);
      mbar_init(b_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(acc_full(t), 1);
      mbar_init(acc_empty(t), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpProducer) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && nkey > 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      mbar_arrive_expect_tx(bar_q, gpc * kQTile);
      for (int gl = 0; gl < gpc; ++gl)
        for (int pn = 0; pn < T::kPanels; ++pn)
          tma_load_3d(sQ + gl * kQTile + pn * kQPanel, &map_q, bar_q, pn * 64, g0 + gl,
                      qb * kBlock);
      // The last tile of an odd count also carries block qb (or rows past L, zero-filled);
      // those scores are never read.
      bool ok = true;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int stage = t % ns, use = t / ns;
        if (*abort_flag || !mbar_wait(b_empty(stage), (use & 1) ^ 1, a.wait_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(b_full(stage), kKTile);
        for (int pn = 0; pn < T::kPanels; ++pn)
          tma_load_2d(sK + stage * kKTile + pn * kKPanel, &map_k, b_full(stage), pn * 64,
                      t * kIndexKeyTile);
        ++issued;
      }
      if (!ok) {
        report_status(a.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // Drain (bounded by the default limit, not the caller's): after an abort the newest load
      // of every stage may still be in flight; the CTA stays until it has landed.
      if (*abort_flag) {
        mbar_wait(bar_q, 0, kDefaultWaitNs);
        for (int it = (issued > ns ? issued - ns : 0); it < issued; ++it)
          mbar_wait(b_full(it % ns), (it / ns) & 1, kDefaultWaitNs);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && nkey > 0) {
      bool ok = mbar_wait(bar_q, 0, a.wait_ns);
      for (int t = 0; ok && t < ntiles; ++t) {
        const int stage = t % ns, suse = t / ns;
        if (*abort_flag || !mbar_spin(b_full(stage), suse & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        const uint32_t kst = sK + stage * kKTile;
        for (int gl = 0; gl < gpc; ++gl) {
          const int u = t * gpc + gl, slot = u & 1;
          if (*abort_flag || !mbar_spin(acc_empty(slot), ((u >> 1) & 1) ^ 1, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + slot * kIndexKeyTile;
          const uint32_t qt = sQ + gl * kQTile;
#pragma unroll
          for (int kk = 0; kk < T::kSteps; ++kk) {
            const uint32_t col = (kk & 3) * 32;
            const uint64_t ad = sdesc_sw128(qt + (kk >> 2) * kQPanel + col, 16, 1024);
            const uint64_t bd = sdesc_sw128(kst + (kk >> 2) * kKPanel + col, 16, 1024);
            if (kF8)
              mma_f8_ss(d, ad, bd, T::kIdesc, kk > 0);
            else
              mma_bf16_ss(d, ad, bd, T::kIdesc, kk > 0);
          }
          mma_commit(acc_full(slot));
        }
        if (!ok) break;
        mma_commit(b_empty(stage));
      }
      if (!ok) {
        report_status(a.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // every MMA this thread issued has finished before the TMEM is released
      mma_commit(drain_bar);
      mbar_wait(drain_bar, 0, kDefaultWaitNs);
    }
  } else {
    // ------------- epilogue warpgroup e: slot e -> max-pool -> top-k -------------
    const int e = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t acc = tmem + lane_base + e * kIndexKeyTile;
    TopList list;
    list.clear();
    bool ok = true;
    for (int u = e; ok && u < nunits; u += 2) {
      const int t = u / gpc;
      // warp-uniform outcome, so the .sync.aligned TMEM loads below never see a split warp
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full(e), (u >> 1) & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // The block maxima come out of the TMEM loads themselves (tcgen05.ld.red .max over each
      // load's 32 columns); the loaded values are not needed.  Two loads in flight per wait (a
      // third would not fit the registers a thread may hold); the slot is released as soon as
      // the last load has landed.
      float mx[2] = {-__int_as_float(0x7f800000), -__int_as_float(0x7f800000)};
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {  // columns [64c, 64c + 64): block c / 2
        uint32_t v0[32], v1[32];
        float a0, a1;
        tmem_ld32_max(acc + c * 64, v0, a0);
        tmem_ld32_max(acc + c * 64 + 32, v1, a1);
        tmem_ld_wait();
        const float m = fmaxf(a0, a1);
        if (c < 2)
          mx[0] = fmaxf(mx[0], m);
        else
          mx[1] = fmaxf(mx[1], m);
      }
      tc_fence_before();
      mbar_arrive(acc_empty(e));
      list.insert(mx[0], a.kb0 + 2 * t);
      if (2 * t + 1 < nkey) list.insert(mx[1], a.kb0 + 2 * t + 1);
      const int64_t ib = static_cast<int64_t>(qb) * kBlock + row;
      if (a.block_scores && ib < a.L) {
        float* bs = a.block_scores +
                    (static_cast<size_t>(g0 + (gpc == 2 ? e : 0)) * a.L + ib) * a.nb + a.kb0 +
                    2 * t;
        bs[0] = mx[0];
        if (2 * t + 1 < nkey) bs[1] = mx[1];
      }
    }
    if (!ok) {
      report_status(a.status, kStatusTimeout);
      *abort_flag = 1;
    }
    if (gpc == 1) {
      // Both warpgroups are past their last score tile, so every MMA and every key load is done
      // and the first key stage can carry warpgroup 1's list to warpgroup 0.
      named_barrier(2, 256);
      float* xs = reinterpret_cast<float*>(smem + (sK - sQ));
      int32_t* xb = reinterpret_cast<int32_t*>(xs + kListMax * 128);
      if (e == 1 && ok && !*abort_flag) {
#pragma unroll
        for (int p = 0; p < kListMax; ++p) {
          xs[p * 128 + row] = list.s[p];
          xb[p * 128 + row] = list.b[p];
        }
      }
      named_barrier(2, 256);
      if (e == 0) {
#pragma unroll
        for (int p = 0; p < kListMax; ++p) list.insert(xs[p * 128 + row], xb[p * 128 + row]);
      }
    }
    const int64_t i = static_cast<int64_t>(qb) * kBlock + row;
    if ((gpc == 2 || e == 0) && ok && !*abort_flag && i < a.L) {
      const int n = min(a.k - 1, nkey);
      const int g = g0 + (gpc == 2 ? e : 0);
#if defined(MSA_DEBUG_CHECKS)
      // checked build: the kept blocks are blocks this CTA scored (at most one failure recorded
      // per row), and the row belongs to a group of the call
      MSA_IN_RANGE(a.status, kSiteIndexRow, g, a.G, i);
#pragma unroll
      for (int p = 0; p < kListMax; ++p)
        if (p < n && !MSA_IN_RANGE(a.status, kSiteIndexRow, list.b[p] - a.kb0, nkey, i)) break;
#endif
      if (a.cand_block) {  // the list is in rank order
        const size_t off = (static_cast<size_t>(g) * a.L + i) * (a.k - 1);
        write_cand_row(list, n, a.k - 1, a.cand_score + off, a.cand_block + off);
      } else {
        list.truncate_and_sort_by_block(n);
        const size_t off = (static_cast<size_t>(g) * a.L + i) * a.k;
        write_sel_row(list, n, qb, a.k, a.sel + off, a.sel_score ? a.sel_score + off : nullptr);
      }
    }
    if (a.block_scores && (gpc == 2 || e == 0) && ok && !*abort_flag) {
      // Row tails: +inf at the local block (never scored), -inf after it (not causal).  The
      // warp walks its 32 rows with the lanes along the columns, so each store is contiguous.
      const int g = g0 + (gpc == 2 ? e : 0);
      const int64_t r0 = static_cast<int64_t>(qb) * kBlock + (warp & 3) * 32;
      for (int r = 0; r < 32 && r0 + r < a.L; ++r) {
        float* bs = a.block_scores + (static_cast<size_t>(g) * a.L + r0 + r) * a.nb;
        for (int b = qb + lane; b < a.nb; b += 32)
          bs[b] = b == qb ? __int_as_float(0x7f800000) : -__int_as_float(0x7f800000);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool kF8>
size_t smem_bytes(int gpc, int ns) {
  return 1024 + static_cast<size_t>(gpc) * IdxTiles<kF8>::kQTile +
         static_cast<size_t>(ns) * IdxTiles<kF8>::kKTile + kBarBytes;
}

template <bool kF8>
cudaError_t launch(const CUtensorMap& map_q, const CUtensorMap& map_k, int64_t L, int G, int k,
                   int32_t* sel, float* sel_score, float* block_scores, int32_t* status,
                   uint64_t wait_ns, int kb0, int kb1, float* cand_score, int32_t* cand_block,
                   cudaStream_t stream) {
  const int nb = static_cast<int>((L + kBlock - 1) / kBlock);
  const int gpc = (G % 2 == 0) ? 2 : 1;  // groups per CTA
  int ns = IdxTiles<kF8>::kMaxStages;    // key stages
  while (ns > 1 && smem_bytes<kF8>(gpc, ns) > 232448) --ns;
  const size_t smem = smem_bytes<kF8>(gpc, ns);
  cudaError_t e = cudaFuncSetAttribute(index_select_prefill_kernel<kF8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  IndexPrefillArgs a{L,       G,       gpc,  k,   nb,         ns,         sel,
                     sel_score, block_scores, status, wait_ns, kb0, kb1, cand_score,
                     cand_block};
  return launch_pdl(index_select_prefill_kernel<kF8>, dim3(nb * (G / gpc)), dim3(kIndexThreads),
                    smem, stream, map_q, map_k, a);
}

}  // namespace

cudaError_t launch_index_select_prefill(const CUtensorMap& map_q, const CUtensorMap& map_k,
                                        int64_t L, int G, int k, bool fp8, int32_t* sel,
                                        float* sel_score, float* block_scores, int32_t* status,
                                        uint64_t wait_ns, cudaStream_t stream, int kb0, int kb1,
                                        float* cand_score, int32_t* cand_block) {
  return fp8 ? launch<true>(map_q, map_k, L, G, k, sel, sel_score, block_scores, status, wait_ns,
                            kb0, kb1, cand_score, cand_block, stream)
             : launch<false>(map_q, map_k, L, G, k, sel, sel_score, block_scores, status,
                             wait_ns, kb0, kb1, cand_score, cand_block, stream);
}

}  // namespace msa
