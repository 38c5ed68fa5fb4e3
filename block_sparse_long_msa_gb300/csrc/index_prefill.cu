// Index branch for prefill, fused: raw index scores (tcgen05 GEMM) -> 128-token block max-pool
// -> per-group top-(k-1) of the earlier blocks -> + local block.  The L x L score matrix never
// leaves the SM: each 128 x 128 score tile lives in TMEM only until its row maxima are taken.
//
// Method: "MiniMax M3 算力省 20 倍", section 二 (index scores over the causal window, max-pooling,
// per-group top-k, forced local block) and section 四 (exp-free top-k: ranking uses raw scores).
//
// One CTA owns one query block qb (128 queries) for all G groups: the G index-query tiles stay
// resident in shared memory while the key blocks 0..qb-1 stream through a TMA ring, so every
// key tile fetched from L2 feeds G MMAs.  Roles:
//   warp 0      TMA producer (q_idx tiles once, then k_idx blocks)
//   warp 1      TMEM owner + single-thread tcgen05.mma issuer
//   warps 4..   one epilogue warpgroup per group; thread r owns query row r: it pulls its 128
//               scores of a key block out of TMEM, max-pools them, and keeps a register top-15.
// Key blocks arrive in ascending order, so a strict "ranks before" test gives the tie rule
// (higher score, then lower block id) without extra state.
#include "common.cuh"
#include "launch.h"

namespace msa {

namespace {

constexpr uint32_t kTile = 32768;   // 128 rows x 128 bf16
constexpr uint32_t kPanel = 16384;  // 128 rows x 64 bf16 (one 128-byte swizzle panel)
constexpr int kAccSlots = 4;        // TMEM accumulator slots of 128 fp32 columns (512 total)
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);

struct IndexPrefillArgs {
  int64_t L;
  int32_t G, k, nb, ns;
  int32_t* sel;
  float* sel_score;
  int32_t* status;
  uint64_t wait_ns;
};

__global__ void __launch_bounds__(640, 1)
    index_select_prefill_kernel(const __grid_constant__ CUtensorMap map_q,
                                const __grid_constant__ CUtensorMap map_k, IndexPrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int G = a.G, ns = a.ns;
  const int S = kAccSlots / G;  // accumulator slots per group
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + G * kTile;
  const uint32_t bars = sB + ns * kTile;
  const uint32_t bar_a = bars;
  auto b_full = [&](int s) { return bars + 8 + 8 * s; };
  auto b_empty = [&](int s) { return bars + 72 + 8 * s; };
  auto acc_full = [&](int t) { return bars + 136 + 8 * t; };
  auto acc_empty = [&](int t) { return bars + 168 + 8 * t; };
  const uint32_t drain_bar = bars + 200;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + (bars - sA) + 208);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + (bars - sA) + 212);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = a.nb - 1 - static_cast<int>(blockIdx.x);  // heaviest query blocks first
  const int nkey = qb;                                      // key blocks 0..qb-1

  if (threadIdx.x == 0) {
    mbar_init(bar_a, 1);
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
        tma_load_3d(sA + g * kTile, &map_q, bar_a, 0, g, qb * kBlock);
        tma_load_3d(sA + g * kTile + kPanel, &map_q, bar_a, 64, g, qb * kBlock);
      }
      int issued = 0;
      for (int j = 0; j < nkey; ++j) {
        const int stage = j % ns, use = j / ns;
        if (*abort_flag || !mbar_wait(b_empty(stage), (use & 1) ^ 1, a.wait_ns)) {
          report_status(a.status, kStatusTimeout);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(b_full(stage), kTile);
        tma_load_2d(sB + stage * kTile, &map_k, b_full(stage), 0, j * kBlock);
        tma_load_2d(sB + stage * kTile + kPanel, &map_k, b_full(stage), 64, j * kBlock);
        ++issued;
      }
      // Drain: the newest load of every stage may still be in flight only after an abort;
      // waiting on it (bounded) keeps the CTA alive until the copy has landed.
      if (*abort_flag) {
        mbar_wait(bar_a, 0, a.wait_ns);
        for (int it = (issued > ns ? issued - ns : 0); it < issued; ++it)
          mbar_wait(b_full(it % ns), (it / ns) & 1, a.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && nkey > 0) {
      bool ok = mbar_wait(bar_a, 0, a.wait_ns);
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
          const int slot = g * S + (j % S), use = j / S;
          if (*abort_flag || !mbar_wait(acc_empty(slot), (use & 1) ^ 1, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + slot * 128;
          const uint32_t ag = sA + g * kTile;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
            mma_bf16_ss(d, sdesc_sw128(ag + off, 16, 1024), sdesc_sw128(bstage + off, 16, 1024),
                        kIdescS, kk > 0);
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
      mbar_wait(drain_bar, 0, a.wait_ns);
    }
  } else if (warp >= 4) {
    // ---------------- epilogue: max-pool + top-k, one warpgroup per group ----------------
    const int g = (warp >> 2) - 1;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    TopList list;
    list.clear();
    bool ok = true;
    for (int j = 0; j < nkey; ++j) {
      const int slot = g * S + (j % S), use = j / S;
      // warp-uniform outcome, so the .sync.aligned TMEM loads below never see a split warp
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full(slot), use & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float mx = -__int_as_float(0x7f800000);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + slot * 128 + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q) mx = fmaxf(mx, __uint_as_float(v[q]));
      }
      tc_fence_before();
      mbar_arrive(acc_empty(slot));
      list.insert(mx, j);
    }
    if (!ok) {
      report_status(a.status, kStatusTimeout);
      *abort_flag = 1;
    }
    const int64_t i = static_cast<int64_t>(qb) * kBlock + row;
    if (ok && !*abort_flag && i < a.L) {
      const int n = min(a.k - 1, nkey);
      list.truncate_and_sort_by_block(n);
      const size_t off = (static_cast<size_t>(g) * a.L + i) * a.k;
      write_sel_row(list, n, qb, a.k, a.sel + off, a.sel_score ? a.sel_score + off : nullptr);
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

size_t index_prefill_smem_bytes(int G, int ns) { return 1024 + (G + ns) * kTile + 256; }

cudaError_t launch_index_select_prefill(const CUtensorMap& map_q, const CUtensorMap& map_k,
                                        int64_t L, int G, int k, int32_t* sel, float* sel_score,
                                        int32_t* status, uint64_t wait_ns, cudaStream_t stream) {
  const int nb = static_cast<int>((L + kBlock - 1) / kBlock);
  int ns = 4;
  while (ns > 2 && index_prefill_smem_bytes(G, ns) > 232448) --ns;
  const size_t smem = index_prefill_smem_bytes(G, ns);
  cudaError_t e = cudaFuncSetAttribute(index_select_prefill_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  IndexPrefillArgs a{L, G, k, nb, ns, sel, sel_score, status, wait_ns};
  index_select_prefill_kernel<<<nb, 128 + 128 * G, smem, stream>>>(map_q, map_k, a);
  return cudaGetLastError();
}

}  // namespace msa
