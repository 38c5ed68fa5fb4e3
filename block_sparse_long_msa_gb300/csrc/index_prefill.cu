// Index branch for prefill, fused: raw index scores (tcgen05 GEMM) -> 128-token block max-pool
// -> per-group top-(k-1) of the earlier blocks -> + local block.  The L x L score matrix never
// leaves the SM: each 128 x 128 score tile lives in TMEM only until its row maxima are taken.
//
// Method: "MiniMax M3 算力省 20 倍", section 二 (index scores over the causal window, max-pooling,
// per-group top-k, forced local block) and section 四 (exp-free top-k: ranking uses raw scores).
//
// One CTA owns one query block qb (128 queries) for all G groups: the G index-query tiles sit in
// TMEM (the MMA's A operand) while the key blocks 0..qb-1 stream through a 6-deep TMA ring in
// shared memory, so every key tile fetched from L2 feeds G MMAs and shared memory carries only
// the keys.  Roles:
//   warp 0      TMA producer (q_idx tiles once, then k_idx blocks)
//   warp 1      TMEM owner + single-thread tcgen05.mma issuer
//   warps 4..   epilogue warpgroups (two for G >= 2); thread r owns query row r: it moves its
//               index-query rows into TMEM once, then pulls its 128 scores of each key block
//               out of TMEM, max-pools them, and keeps a register top-15 per group.
// Key blocks arrive in ascending order, so a strict "ranks before" test gives the tie rule
// (higher score, then lower block id) without extra state.
#include "common.cuh"
#include "launch.h"

namespace msa {

namespace {

constexpr uint32_t kTile = 32768;   // 128 rows x 128 bf16
constexpr uint32_t kPanel = 16384;  // 128 rows x 64 bf16 (one 128-byte swizzle panel)
constexpr int kAccSlots = 2;        // TMEM accumulators of 128 fp32 columns: columns [0, 256)
constexpr uint32_t kAcolBase = 256; // index-query tiles in TMEM: 64 columns per group
constexpr int kMaxStages = 8;
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);

struct IndexPrefillArgs {
  int64_t L;
  int32_t G, k, nb, ns;
  int32_t* sel;
  float* sel_score;
  int32_t* status;
  uint64_t wait_ns;
};

// Which accumulator slot, and which use of it, the score tile of (key block j, group g) takes.
// G = 1: the two slots alternate over key blocks; G = 2: one slot per group; G = 4: groups
// g and g+2 share slot g & 1.
__device__ __forceinline__ void slot_of(int G, int j, int g, int& slot, int& use) {
  if (G == 1) {
    slot = j & 1;
    use = j >> 1;
  } else if (G == 2) {
    slot = g;
    use = j;
  } else {
    slot = g & 1;
    use = 2 * j + (g >> 1);
  }
}

// Shared memory: ns key stages of 32 KB (the first G of them first carry the index-query tiles on
// their way into TMEM), then the barrier block.
__global__ void __launch_bounds__(384, 1)
    index_select_prefill_kernel(const __grid_constant__ CUtensorMap map_q,
                                const __grid_constant__ CUtensorMap map_k, IndexPrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int G = a.G, ns = a.ns;
  const uint32_t sB = smem_u32(smem);
  const uint32_t bars = sB + ns * kTile;
  const uint32_t bar_a = bars;                                // index-query tiles landed
  const uint32_t a_ready = bars + 8;                          // ... and copied into TMEM
  auto b_full = [&](int s) { return bars + 16 + 8 * s; };     // 8 slots: [16, 80)
  auto b_empty = [&](int s) { return bars + 80 + 8 * s; };    // [80, 144)
  auto acc_full = [&](int t) { return bars + 144 + 8 * t; };  // [144, 160)
  auto acc_empty = [&](int t) { return bars + 160 + 8 * t; }; // [160, 176)
  const uint32_t drain_bar = bars + 176;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + (bars - sB) + 184);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + (bars - sB) + 188);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = a.nb - 1 - static_cast<int>(blockIdx.x);  // heaviest query blocks first
  const int nkey = qb;                                      // key blocks 0..qb-1
  const int n_epi = G == 1 ? 1 : 2;                         // epilogue warpgroups

  if (threadIdx.x == 0) {
    mbar_init(bar_a, 1);
    mbar_init(a_ready, 128);
    for (int s = 0; s < ns; ++s) {
      mbar_init(b_full(s), 1);
      mbar_init(b_empty(s), 1);
    }
    for (int t = 0; t < kAccSlots; ++t) {
      mbar_init(acc_full(t), 1);
      mbar_init(acc_empty(t), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && nkey > 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      mbar_arrive_expect_tx(bar_a, G * kTile);
      for (int g = 0; g < G; ++g) {
        tma_load_3d(sB + g * kTile, &map_q, bar_a, 0, g, qb * kBlock);
        tma_load_3d(sB + g * kTile + kPanel, &map_q, bar_a, 64, g, qb * kBlock);
      }
      // the first G stages are free again once the tiles are in TMEM
      bool ok = mbar_wait(a_ready, 0, a.wait_ns);
      int issued = 0;
      for (int j = 0; ok && j < nkey; ++j) {
        const int stage = j % ns, use = j / ns;
        if (*abort_flag || !mbar_wait(b_empty(stage), (use & 1) ^ 1, a.wait_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(b_full(stage), kTile);
        tma_load_2d(sB + stage * kTile, &map_k, b_full(stage), 0, j * kBlock);
        tma_load_2d(sB + stage * kTile + kPanel, &map_k, b_full(stage), 64, j * kBlock);
        ++issued;
      }
      if (!ok) {
        report_status(a.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // Drain (bounded by the default limit, not the caller's): the newest load of every stage
      // may still be in flight only after an abort; the CTA stays until it has landed.
      if (*abort_flag) {
        mbar_wait(bar_a, 0, kDefaultWaitNs);
        for (int it = (issued > ns ? issued - ns : 0); it < issued; ++it)
          mbar_wait(b_full(it % ns), (it / ns) & 1, kDefaultWaitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && nkey > 0) {
      bool ok = mbar_wait(a_ready, 0, a.wait_ns);
      tc_fence_after();
      for (int j = 0; ok && j < nkey; ++j) {
        const int stage = j % ns, suse = j / ns;
        if (*abort_flag || !mbar_wait(b_full(stage), suse & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t bstage = sB + stage * kTile;
        for (int g = 0; g < G; ++g) {
          int slot, use;
          slot_of(G, j, g, slot, use);
          if (*abort_flag || !mbar_wait(acc_empty(slot), (use & 1) ^ 1, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + slot * 128;
          const uint32_t at = tmem + kAcolBase + g * 64;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
            mma_f16_ts(d, at + kk * 8, sdesc_sw128(bstage + off, 16, 1024), kIdescS, kk > 0);
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
  } else if (warp >= 4 && warp < 4 + 4 * n_epi) {
    // ------------- epilogue: max-pool + top-k; warpgroup e takes the groups g = e (mod 2) -------
    const int e = (warp >> 2) - 1;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    if (e == 0 && nkey > 0) {
      // index-query tiles: shared memory (swizzled, from TMA) -> TMEM columns [256 + 64 g, +64)
      const bool landed = __all_sync(0xffffffffu, mbar_wait(bar_a, 0, a.wait_ns));
      if (!landed) {
        report_status(a.status, kStatusTimeout);
        *abort_flag = 1;
      }
      for (int g = 0; landed && g < G; ++g) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 x = ld_shared_v4(sB + g * kTile + sw128_offset(row, h * 64 + c * 8, 128));
            r[4 * c] = x.x;
            r[4 * c + 1] = x.y;
            r[4 * c + 2] = x.z;
            r[4 * c + 3] = x.w;
          }
          tmem_st32(tmem + lane_base + kAcolBase + g * 64 + h * 32, r);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(a_ready);
    }
    TopList list0, list1;  // groups e and e + 2
    list0.clear();
    list1.clear();
    bool ok = true;
    const int steps_per_j = G == 4 ? 2 : 1;
    for (int j = 0; ok && j < nkey; ++j) {
      for (int q = 0; q < steps_per_j; ++q) {
        const int g = G == 1 ? 0 : e + 2 * q;
        int slot, use;
        slot_of(G, j, g, slot, use);
        // warp-uniform outcome, so the .sync.aligned TMEM loads below never see a split warp
        if (!__all_sync(0xffffffffu, mbar_wait(acc_full(slot), use & 1, a.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float mx = -__int_as_float(0x7f800000);
#pragma unroll 1
        for (int c = 0; c < 4; c += 2) {
          uint32_t v0[32], v1[32];
          tmem_ld32(tmem + lane_base + slot * 128 + c * 32, v0);
          tmem_ld32(tmem + lane_base + slot * 128 + c * 32 + 32, v1);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < 32; ++t)
            mx = fmaxf(mx, fmaxf(__uint_as_float(v0[t]), __uint_as_float(v1[t])));
        }
        tc_fence_before();
        mbar_arrive(acc_empty(slot));
        if (q == 0) list0.insert(mx, j);
        else list1.insert(mx, j);
      }
    }
    if (!ok) {
      report_status(a.status, kStatusTimeout);
      *abort_flag = 1;
    }
    const int64_t i = static_cast<int64_t>(qb) * kBlock + row;
    if (ok && !*abort_flag && i < a.L) {
      const int n = min(a.k - 1, nkey);
      {
        const int g = G == 1 ? 0 : e;
        list0.truncate_and_sort_by_block(n);
        const size_t off = (static_cast<size_t>(g) * a.L + i) * a.k;
        write_sel_row(list0, n, qb, a.k, a.sel + off, a.sel_score ? a.sel_score + off : nullptr);
      }
      if (steps_per_j == 2) {
        const int g = e + 2;
        list1.truncate_and_sort_by_block(n);
        const size_t off = (static_cast<size_t>(g) * a.L + i) * a.k;
        write_sel_row(list1, n, qb, a.k, a.sel + off, a.sel_score ? a.sel_score + off : nullptr);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t index_prefill_smem_bytes(int G, int ns) {
  (void)G;
  return 1024 + static_cast<size_t>(ns) * kTile + 256;
}

cudaError_t launch_index_select_prefill(const CUtensorMap& map_q, const CUtensorMap& map_k,
                                        int64_t L, int G, int k, int32_t* sel, float* sel_score,
                                        int32_t* status, uint64_t wait_ns, cudaStream_t stream) {
  const int nb = static_cast<int>((L + kBlock - 1) / kBlock);
  int ns = 6;  // key stages; the first G also stage the index-query tiles
  while (ns > 4 && index_prefill_smem_bytes(G, ns) > 232448) --ns;
  const size_t smem = index_prefill_smem_bytes(G, ns);
  cudaError_t e = cudaFuncSetAttribute(index_select_prefill_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  IndexPrefillArgs a{L, G, k, nb, ns, sel, sel_score, status, wait_ns};
  const int threads = 128 + 128 * (G == 1 ? 1 : 2);
  index_select_prefill_kernel<<<nb, threads, smem, stream>>>(map_q, map_k, a);
  return cudaGetLastError();
}

}  // namespace msa
