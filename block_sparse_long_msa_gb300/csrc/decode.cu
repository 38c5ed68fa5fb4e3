// Paged decode: one query per sequence at position n-1 over a cache of 128-token pages.
//
//   index branch ("MiniMax M3 算力省 20 倍", section 二; paged decode as named on the page about
//   serving MSA): every index-key page strictly before the query's page is scored against the
//   sequence's G index queries and max-pooled, then each (sequence, group) keeps its top-(k-1)
//   blocks plus the local block (section 四: exp-free top-k, lanes each stream 1/32 of the row
//   and their lists are merged with warp shuffles).
//   main branch: exact softmax attention of the 16 query heads of a group over the selected
//   pages (causal inside the local page), one partial per (sequence, group, slot), merged by a
//   log-sum-exp combine.
//
// The scan is the dominant stream of this step (every index key of every sequence, 32 KiB per
// page in bf16, 16 KiB in e4m3); it is fed by TMA into a deep shared-memory ring and scored by
// tcgen05 with the page as the 128-row A operand, so the SM's issue slots stay free for the
// max-pool.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace msa {

namespace {

constexpr int kHeads = 16;  // query heads per group
constexpr uint32_t kPanel = 16384;  // 128 rows x 128 bytes: one 128-byte-swizzled panel
// Scan stage: one index-key page (128 keys, K-major, 128-byte swizzle: two 64-element panels
// per bf16 row, one per e4m3 row) and a 16-row index-query tile (rows G..15 zero).  Every MMA
// step covers 32 bytes of K: 8 bf16 steps or 4 e4m3 steps for K = 128.
template <bool kF8>
struct ScanTiles {
  static constexpr uint32_t kEsz = kF8 ? 1 : 2;
  static constexpr uint32_t kKeys = kBlock * kDim * kEsz;      // 32 KB bf16, 16 KB e4m3
  static constexpr uint32_t kQRows = 16 * kDim * kEsz;         // 4 KB bf16, 2 KB e4m3
  static constexpr uint32_t kQPanel = 16 * 128;
  static constexpr uint32_t kStage = kKeys + kQRows;
  static constexpr int kPanels = kF8 ? 1 : 2;
  static constexpr int kSteps = kF8 ? 4 : 8;
  static constexpr int kStages = kF8 ? 4 : 3;  // 72 KiB (e4m3) or 108 KiB (bf16) per CTA
  static constexpr uint32_t kIdesc = kF8 ? idesc_e4m3_f32(128, 16)
                                         : idesc_bf16_f32(128, 16, false, false);
};
constexpr int kScanMaxStages = 12;
constexpr int kScanSlots = 8;                  // TMEM accumulators of 16 columns
// barrier block after the stages: full[], empty[], acc_full[8], acc_empty[8], drain, then the
// TMEM base address, the abort flag and the CTA's page range
constexpr uint32_t kScanBarFull = 0, kScanBarEmpty = 96, kScanBarAccFull = 192,
                   kScanBarAccEmpty = 256, kScanBarDrain = 320, kScanTmemSlot = 328,
                   kScanAbort = 332, kScanWalk = 336, kScanBarBytes = 512;
static_assert(kScanBarFull + 8 * kScanMaxStages <= kScanBarEmpty, "scan barriers");
static_assert(kScanBarEmpty + 8 * kScanMaxStages <= kScanBarAccFull, "scan barriers");
static_assert(kScanBarAccFull + 8 * kScanSlots <= kScanBarAccEmpty, "scan barriers");
static_assert(kScanBarAccEmpty + 8 * kScanSlots <= kScanBarDrain, "scan barriers");
static_assert(kScanAbort + 4 <= kScanWalk, "scan barriers");
static_assert(kScanWalk + 12 <= kScanBarBytes, "scan barriers");
template <bool kF8>
constexpr uint32_t scan_smem() {
  return ScanTiles<kF8>::kStages * ScanTiles<kF8>::kStage + kScanBarBytes + 1024;
}
static_assert(ScanTiles<false>::kStages <= kScanMaxStages && scan_smem<false>() <= 232448,
              "scan shared memory");
static_assert(ScanTiles<true>::kStages <= kScanMaxStages && scan_smem<true>() <= 232448,
              "scan shared memory");
// Several scan CTAs share an SM (233,472 bytes of shared memory, 1 KB of it reserved per CTA), so
// each SM runs independent page pipelines: two with bf16 pages, three with the half-size e4m3
// pages (at 56 registers a thread, the register file's share of three CTAs).
template <bool kF8>
constexpr int scan_ctas_per_sm() { return kF8 ? 3 : 2; }
static_assert(scan_ctas_per_sm<false>() * (scan_smem<false>() + 1024) <= 233472 &&
                  scan_ctas_per_sm<true>() * (scan_smem<true>() + 1024) <= 233472,
              "scan CTAs per SM");

struct ScanArgs {
  const int32_t* page_table;
  const int32_t* seq_lens;
  int32_t batch, max_pages, num_pages, G;
  int32_t kb0, kb1;  // logical blocks scanned: [kb0, kb1) (0, max_pages: all of them)
  float4* scores;    // [batch][G][max_pages]: per-warp maxima of the 4 epilogue warps
  int32_t* status;
  uint64_t wait_ns;
};

// Index pages scored for sequence s: those of [kb0, kb1) strictly before the query's page.
__device__ __forceinline__ int scan_pages(const ScanArgs& a, int s) {
  const int n = a.seq_lens[s];
  const int before = n > 0 ? min((n - 1) / kBlock, a.max_pages) : 0;
  return max(0, min(before, a.kb1) - a.kb0);
}

// The pages of all sequences, concatenated in (sequence, block) order, are split into equal
// contiguous ranges, one per CTA.  One warp finds the CTA's first page with warp prefix sums over
// the sequence lengths; every role then walks the range identically.
__device__ void scan_range(const ScanArgs& a, int lane, int* out /* s0, b0, count */) {
  long long total = 0;
  for (int s0 = 0; s0 < a.batch; s0 += 32) {
    const int s = s0 + lane;
    int c = s < a.batch ? scan_pages(a, s) : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    total += c;
  }
  const long long p0 = total * blockIdx.x / gridDim.x;
  const long long p1 = total * (blockIdx.x + 1) / gridDim.x;
  long long before = 0;  // pages of the sequences before the current group of 32
  int s_first = a.batch, b_first = 0;
  for (int s0 = 0; s0 < a.batch && s_first == a.batch; s0 += 32) {
    const int s = s0 + lane;
    const int c = s < a.batch ? scan_pages(a, s) : 0;
    int incl = c;  // inclusive prefix within the group
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const long long start = before + incl - c;
    // the sequence whose pages contain p0 (first lane whose range reaches past it)
    const unsigned hit = __ballot_sync(0xffffffffu, c > 0 && start <= p0 && p0 < start + c);
    if (hit) {
      const int l = __ffs(hit) - 1;
      s_first = s0 + l;
      b_first = static_cast<int>(p0 - __shfl_sync(0xffffffffu, start, l));
    }
    before += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    out[0] = s_first;
    out[1] = b_first;
    out[2] = static_cast<int>(p1 - p0);
  }
}

struct PageWalk {
  int s, b, left, ns;  // b counts the scanned pages of sequence s, from 0
  __device__ __forceinline__ void init(const ScanArgs& a, const volatile int* r) {
    s = r[0];
    b = r[1] - 1;
    left = r[2];
    ns = left > 0 ? scan_pages(a, s) : 0;
  }
  // Advances to the next page of the range; returns its logical block id, or -1 at the end.
  __device__ __forceinline__ int next(const ScanArgs& a) {
    if (left <= 0) return -1;
    --left;
    ++b;
    while (b >= ns) {  // on to the next sequence that has pages
      ++s;
      b = 0;
      if (!MSA_IN_RANGE(a.status, kSiteDecodePage, s, a.batch, s)) {  // checked build only
        left = 0;
        return -1;
      }
      ns = scan_pages(a, s);
    }
    return a.kb0 + b;
  }
};

// Maximum of v over the 32 lanes of the (converged) warp, in one instruction (redux.sync with
// .f32, sm_100 family); a NaN operand is ignored as in fmaxf.
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Warps: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2 finds the CTA's page range, 4-11 two
// epilogue groups taking alternate pages (a page's 128 keys are the 128 TMEM lanes, one warp per
// quarter), so two pages' reductions are in flight.
constexpr int kScanThreads = 384;

template <bool kF8>
__global__ void __launch_bounds__(kScanThreads, scan_ctas_per_sm<kF8>())
    decode_scan_kernel(const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_q, ScanArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  using T = ScanTiles<kF8>;
  constexpr int kScanStages = T::kStages;
  constexpr uint32_t kScanStage = T::kStage;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(smem);
  const uint32_t bars = base + kScanStages * kScanStage;
  auto full = [&](int s) { return bars + kScanBarFull + 8 * s; };
  auto empty = [&](int s) { return bars + kScanBarEmpty + 8 * s; };
  auto acc_full = [&](int t) { return bars + kScanBarAccFull + 8 * t; };
  auto acc_empty = [&](int t) { return bars + kScanBarAccEmpty + 8 * t; };
  const uint32_t drain_bar = bars + kScanBarDrain;
  volatile uint32_t* tmem_slot =
      reinterpret_cast<volatile uint32_t*>(smem + kScanStages * kScanStage + kScanTmemSlot);
  volatile int32_t* abort_flag =
      reinterpret_cast<volatile int32_t*>(smem + kScanStages * kScanStage + kScanAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // rows G..15 of every stage's query tile stay zero (TMA writes rows 0..G-1 only)
  for (int st = 0; st < kScanStages; ++st) {
    uint32_t* qt = reinterpret_cast<uint32_t*>(smem + st * kScanStage + T::kKeys);
    for (int w = threadIdx.x; w < static_cast<int>(T::kQRows / 4); w += blockDim.x) qt[w] = 0;
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kScanStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int t = 0; t < kScanSlots; ++t) {
      mbar_init(acc_full(t), 1);
      mbar_init(acc_empty(t), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  volatile int* walk = reinterpret_cast<volatile int*>(smem + kScanStages * kScanStage + kScanWalk);
  if (warp == 2) scan_range(a, lane, const_cast<int*>(walk));
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_q);
      // Page ids are read 8 pages ahead (a batch of independent loads while the previous batch
      // is issued), so the page-table latency stays off the issue path.
      PageWalk w;
      w.init(a, walk);
      auto fetch8 = [&](int (&pid)[8], int (&sq)[8]) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int b = w.next(a);
          sq[j] = b >= 0 ? w.s : -1;
          pid[j] = b >= 0 ? a.page_table[static_cast<size_t>(w.s) * a.max_pages + b] : 0;
        }
      };
      int pa[8], sa[8], pb[8], sb8[8];
      fetch8(pa, sa);
      int p = 0;
      bool more = sa[0] >= 0;
      while (more) {
        fetch8(pb, sb8);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (sa[j] < 0 || *abort_flag) {
            more = false;
            break;
          }
          const int st = p % kScanStages;
          if (!mbar_wait(empty(st), ((p / kScanStages) & 1) ^ 1, a.wait_ns)) {
            report_status(a.status, kStatusTimeout);
            *abort_flag = 1;
            more = false;
            break;
          }
          int page = pa[j];
          if (page < 0 || page >= a.num_pages) {
            report_status(a.status, kStatusBounds);
            page = 0;  // keep the pipeline in step; the status word marks the result invalid
          }
          const uint32_t sbase = base + st * kScanStage;
          mbar_arrive_expect_tx(full(st), T::kKeys + a.G * kDim * T::kEsz);
          for (int pn = 0; pn < T::kPanels; ++pn) {
            tma_load_2d(sbase + pn * kPanel, &map_k, full(st), pn * 64, page * kBlock);
            tma_load_2d(sbase + T::kKeys + pn * T::kQPanel, &map_q, full(st), pn * 64,
                        sa[j] * a.G);
          }
          ++p;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          pa[j] = pb[j];
          sa[j] = sb8[j];
        }
        more = more && sa[0] >= 0;
      }
      // Drain (bounded by the default limit, not the caller's): after an abort the newest load
      // of every stage may still be in flight; the CTA stays until it has landed.
      if (*abort_flag) {
        for (int x = (p > kScanStages ? p - kScanStages : 0); x < p; ++x)
          mbar_wait(full(x % kScanStages), (x / kScanStages) & 1, kDefaultWaitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      PageWalk w;
      w.init(a, walk);
      int p = 0;
      bool ok = true;
      for (int b = w.next(a); b >= 0; b = w.next(a), ++p) {
        const int st = p % kScanStages, slot = p % kScanSlots;
        if (*abort_flag || !mbar_wait(full(st), (p / kScanStages) & 1, a.wait_ns) ||
            !mbar_wait(acc_empty(slot), ((p / kScanSlots) & 1) ^ 1, a.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sb = base + st * kScanStage;
#pragma unroll
        for (int kk = 0; kk < T::kSteps; ++kk) {
          const uint64_t ad = sdesc_sw128(sb + (kk >> 2) * kPanel + (kk & 3) * 32, 16, 1024);
          const uint64_t bd =
              sdesc_sw128(sb + T::kKeys + (kk >> 2) * T::kQPanel + (kk & 3) * 32, 16, 1024);
          if (kF8)
            mma_f8_ss(tmem + slot * 16, ad, bd, T::kIdesc, kk > 0);
          else
            mma_bf16_ss(tmem + slot * 16, ad, bd, T::kIdesc, kk > 0);
        }
        mma_commit(acc_full(slot));
        mma_commit(empty(st));
      }
      if (!ok) {
        report_status(a.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // every MMA this thread issued has finished before the TMEM is released (the default
      // limit, so that a short caller limit cannot cut the drain short)
      mma_commit(drain_bar);
      mbar_wait(drain_bar, 0, kDefaultWaitNs);
    }
  } else if (warp >= 4) {
    // epilogue: thread = key of the page; the warp's max over its 32 keys per group.  Group eg
    // takes the pages p with p % 2 == eg; an even number of slots keeps every slot with one
    // group, which therefore sees each of its slot's phases in order.
    static_assert(kScanSlots % 2 == 0, "scan slots per epilogue group");
    const int eg = (warp - 4) >> 2, ew = (warp - 4) & 3;
    const uint32_t lane_base = static_cast<uint32_t>(ew * 32) << 16;
    PageWalk w;
    w.init(a, walk);
    int p = 0;
    for (int b = w.next(a); b >= 0; b = w.next(a), ++p) {
      if ((p & 1) != eg) continue;
      const int slot = p % kScanSlots;
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full(slot), (p / kScanSlots) & 1, a.wait_ns))) {
        report_status(a.status, kStatusTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      uint32_t v[4];
      tmem_ld4(tmem + lane_base + slot * 16, v);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(acc_empty(slot));
      float m[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) m[g] = warp_max_f32(__uint_as_float(v[g]));
      if (lane < a.G && MSA_IN_RANGE(a.status, kSiteDecodePage, b, a.max_pages, w.s)) {
        float* dst = reinterpret_cast<float*>(
            a.scores + (static_cast<size_t>(w.s) * a.G + lane) * a.max_pages + b);
        dst[ew] = lane == 0 ? m[0] : lane == 1 ? m[1] : lane == 2 ? m[2] : m[3];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ------------------------------------------------------------------------------------------
// Top-k: one CTA of four warps per (sequence, group).  Lane l of warp w streams blocks
// 32w + l, 32w + l + 128, ... into its own rank-ordered list; k-1 rounds of a warp arg-max pop
// each warp's best into shared memory, and warp 0 merges the four lists the same way.  Ranking
// compares (score, block id), so the order in which candidates arrive does not matter.
// ------------------------------------------------------------------------------------------
struct TopkArgs {
  const float4* scores;
  const int32_t* seq_lens;
  int32_t batch, max_pages, G, k;
  int32_t kb0, kb1;   // logical blocks ranked: [kb0, kb1)
  int32_t* sel;       // [G][batch][k]
  float* sel_score;   // optional, same shape
  float* block_scores;  // optional [G][batch][max_pages]: pooled score of every block (+inf
                        // the local one, -inf later ones)
  float* cand_score;    // candidate mode (cand_block set): [G][batch][k-1] in rank order
  int32_t* cand_block;
  int32_t* status;
};

__global__ void __launch_bounds__(128) decode_topk_kernel(TopkArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  __shared__ float cand_s[4][kListMax];
  __shared__ int32_t cand_b[4][kListMax];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x / a.G, g = blockIdx.x % a.G;  // grid = batch * G
  const int n = a.seq_lens[s];
  const bool cand = a.cand_block != nullptr;
  const int width = cand ? a.k - 1 : a.k;  // entries per output row
  int32_t* out = (cand ? a.cand_block : a.sel) + (static_cast<size_t>(g) * a.batch + s) * width;
  float* out_s = cand ? a.cand_score + (static_cast<size_t>(g) * a.batch + s) * width
                 : a.sel_score ? a.sel_score + (static_cast<size_t>(g) * a.batch + s) * a.k
                               : nullptr;
  float* bsrow = a.block_scores
                     ? a.block_scores + (static_cast<size_t>(g) * a.batch + s) * a.max_pages
                     : nullptr;
  const float ninf = -__int_as_float(0x7f800000), pinf = __int_as_float(0x7f800000);
  if (n <= 0 || (n - 1) / kBlock >= a.max_pages) {  // the same outcome for the whole CTA
    if (threadIdx.x == 0) report_status(a.status, kStatusBounds);
    if (warp == 0)
      for (int r = lane; r < width; r += 32) {
        out[r] = -1;
        if (out_s) out_s[r] = ninf;
      }
    if (bsrow)
      for (int b = threadIdx.x; b < a.max_pages; b += 128) bsrow[b] = ninf;
    return;
  }
  const int bi = (n - 1) / kBlock;
  if (bsrow)  // the local block is never scored; later blocks are not causal
    for (int b = bi + threadIdx.x; b < a.max_pages; b += 128) bsrow[b] = b == bi ? pinf : ninf;
  const float4* row = a.scores + (static_cast<size_t>(s) * a.G + g) * a.max_pages;
  // the ranked blocks: [lo, hi), strictly before the local block
  const int lo = a.kb0, hi = min(a.kb1, bi);
  TopList list;
  list.clear();
  // eight loads in flight per lane, then eight inserts
  for (int b0 = lo + warp * 32; b0 < hi; b0 += 8 * 128) {
    float sc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int b = b0 + q * 128 + lane;
      if (b < hi) {
        const float4 v = row[b];
        sc[q] = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int b = b0 + q * 128 + lane;
      if (b < hi) {
        list.insert(sc[q], b);
        if (bsrow) bsrow[b] = sc[q];
      }
    }
  }
  const int take = min(a.k - 1, max(0, hi - lo));
  // r-th round: the warp's r-th best (score, block) reaches every lane; its owner pops it.
  // Empty entries (-inf, INT_MAX) rank last, so a warp with fewer blocks pads with them.
  auto pop_best = [&](float& bs, int& bb) {
    bs = list.s[0];
    bb = list.b[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float os = __shfl_xor_sync(0xffffffffu, bs, o);
      const int ob = __shfl_xor_sync(0xffffffffu, bb, o);
      if (ranks_before(os, ob, bs, bb)) {
        bs = os;
        bb = ob;
      }
    }
    if (list.b[0] == bb) {
#pragma unroll
      for (int q = 0; q + 1 < kListMax; ++q) {
        list.s[q] = list.s[q + 1];
        list.b[q] = list.b[q + 1];
      }
      list.s[kListMax - 1] = ninf;
      list.b[kListMax - 1] = 0x7fffffff;
    }
  };
  for (int r = 0; r < take; ++r) {
    float bs;
    int bb;
    pop_best(bs, bb);
    if (lane == 0) {
      cand_s[warp][r] = bs;
      cand_b[warp][r] = bb;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  list.clear();
  for (int c = lane; c < 4 * take; c += 32)
    list.insert(cand_s[c / take][c % take], cand_b[c / take][c % take]);
  int my_id = 0x7fffffff;
  float my_sc = 0.f;
  for (int r = 0; r < take; ++r) {
    float bs;
    int bb;
    pop_best(bs, bb);
    if (lane == r) {
      my_id = bb;
      my_sc = bs;
    }
  }
  if (cand) {  // lane r holds the r-th ranked block
    for (int r = lane; r < width; r += 32) {
      out[r] = r < take ? my_id : -1;
      out_s[r] = r < take ? my_sc : ninf;
    }
    return;
  }
  // lanes 0..take-1 hold the winners; place each at its rank by block id
  int rank = 0;
  for (int q = 0; q < take; ++q) {
    const int other = __shfl_sync(0xffffffffu, my_id, q);
    rank += other < my_id;
  }
  if (lane < take) {
    out[rank] = my_id;
    if (out_s) out_s[rank] = my_sc;
  }
  for (int r = take + lane; r < a.k; r += 32) {
    out[r] = r == take ? bi : -1;
    if (out_s) out_s[r] = r == take ? pinf : ninf;
  }
}

// ------------------------------------------------------------------------------------------
// Decode attention: one unit per (sequence, group, slot).  A persistent CTA takes a contiguous
// range of units; warp 0 stages each unit's K and V page tiles (TMA, 128-byte swizzle).  The
// staged units go in turn to three groups of four compute warps (warps 1-4, 5-8, 9-12); in a
// group each warp scores 32 keys (S = q K^T with m16n8k16 MMAs, M = the group's 16 heads), the four
// exchange row maxima, sums and their slice of P through shared memory, and then each computes
// O = P V for 32 of the 128 output dimensions over all the page's keys, written straight to the
// partial.
// With an e4m3 K/V cache (kKV8) the pages arrive as 16 KiB e4m3 tiles and both products run in
// fp16 (every e4m3 value is an fp16 value; q is rounded to fp16 once per (sequence, group),
// which is exact for |q| >= 2^-17).  For S each thread loads its B fragments straight from the
// staged e4m3 tile: inside every 16-wide k-step the head dimension is permuted, the same way for
// q and K, so that a thread's four k elements are four adjacent bytes (one 32-bit load, two
// conversions).  V, read transposed by P.V, is widened by each warp for its 32 dimensions into a
// private swizzled fp16 buffer.
// ------------------------------------------------------------------------------------------
struct DecAttnArgs {
  const __nv_bfloat16* q;  // [batch][G*16][128]
  const int32_t* sel;      // [G][batch][k]
  const int32_t* page_table;
  const int32_t* seq_lens;
  int32_t batch, max_pages, num_pages, G, k;
  int32_t units, per_cta;
  float scale_log2;
  float* po;    // [unit][16][128] normalised partial O
  float* plse;  // [unit][16] log-sum-exp (-inf for empty units)
  int32_t* status;
  uint64_t wait_ns;
};

// Shared-memory layout of the decode attention kernel, by K/V storage type.
// Three groups of four compute warps take the staged units in turn, so every SM sub-partition has
// three warps to interleave (each unit's chain of products, exchanges and barriers is latency-
// bound; two groups: e4m3 0.0662 -> 0.0621 ms per step with three).  416 threads leave a thread
// 152 registers: the bf16 instance uses 127, the e4m3 one 128.  Three stages of pages fit beside
// the e4m3 instance's private fp16 V buffers (12 warps x 8 KiB).
template <bool kKV8>
struct DecLayout {
  static constexpr int kGroups = 3;
  static constexpr int kThreads = 32 + kGroups * 128;
  static constexpr int kStages = 3;
  static constexpr uint32_t kTile = kKV8 ? 16384 : 32768;  // one K or V page tile
  static constexpr uint32_t kStage = 2 * kTile;
  // e4m3: per compute warp, V of its 32 dimensions in fp16 (128 rows x 64 B)
  static constexpr uint32_t kPriv = kStages * kStage;
  static constexpr uint32_t kPrivWarp = 8192;
  static constexpr uint32_t kP = kPriv + (kKV8 ? 4 * kGroups * kPrivWarp : 0);
  // Per unit the four warps of a group exchange their row maxima and row sums and the P tile (16
  // rows x 128 keys, 128-byte swizzled panels); two copies per group, by the parity of the
  // group's units, so a warp may start the next unit while another still reads this one's.
  static constexpr uint32_t kPBytes = kHeads * kBlock * 2;
  static constexpr uint32_t kML = kP + kGroups * 2 * kPBytes;
  static constexpr uint32_t kMLGroup = 2 * 2 * 4 * kHeads * 4;  // 2 x (max, sum) x 4 warps x 16
  static constexpr uint32_t kBar = kML + kGroups * kMLGroup;
  static constexpr uint32_t kSmem = kBar + 128 + 1024;
};
constexpr int kDecMaxStages = 4;
constexpr uint32_t kDecBarFull = 0, kDecBarEmpty = 32, kDecAbort = 64;
static_assert(kDecBarFull + 8 * kDecMaxStages <= kDecBarEmpty, "decode attention barriers");
static_assert(kDecBarEmpty + 8 * kDecMaxStages <= kDecAbort, "decode attention barriers");
static_assert(kDecAbort + 4 <= 128, "decode attention barriers");
static_assert(DecLayout<false>::kStages <= kDecMaxStages && DecLayout<true>::kStages <= kDecMaxStages,
              "decode attention stages");
static_assert(DecLayout<false>::kSmem <= 232448, "decode attention shared memory");
static_assert(DecLayout<true>::kSmem <= 232448, "decode attention shared memory (e4m3)");

struct UnitInfo {
  int s, g, b, page, lim;
  bool valid;
};

__device__ __forceinline__ UnitInfo unit_info(const DecAttnArgs& a, int u, bool flag) {
  UnitInfo x;
  x.s = u / (a.G * a.k);
  x.g = (u / a.k) % a.G;
  const int t = u % a.k;
  x.b = a.sel[(static_cast<size_t>(x.g) * a.batch + x.s) * a.k + t];
  const int n = a.seq_lens[x.s];
  const int bi = n > 0 ? (n - 1) / kBlock : -1;
  x.valid = x.b >= 0 && x.b <= bi && x.b < a.max_pages;
  x.page = 0;
  if (x.valid) {
    x.page = a.page_table[static_cast<size_t>(x.s) * a.max_pages + x.b];
    if (x.page < 0 || x.page >= a.num_pages) x.valid = false;
  }
  if (flag && !x.valid && x.b >= 0) report_status(a.status, kStatusBounds);
  x.lim = x.valid ? min(n - 1 - x.b * kBlock, kBlock - 1) : -1;
  return x;
}

__device__ __forceinline__ uint32_t swz(uint32_t tile, int row, int chunk) {
  return tile + (chunk >> 3) * kPanel + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// The 16 x 128 P tile: two 64-key panels of 16 rows x 128 bytes, 16-byte chunks XOR-swizzled by
// row, so the stores of a warp and the ldmatrix reads both spread over all banks.
__device__ __forceinline__ uint32_t dec_p_addr(uint32_t tile, int row, int chunk) {
  return tile + (chunk >> 3) * (kHeads * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// Private fp16 V buffer of a warp (128 keys x its 32 dimensions = 64 B): chunk c (0..3) of key
// row r, XOR-ed with bits 1..2 of the row (8 consecutive rows then cover all 32 banks).
__device__ __forceinline__ uint32_t vpriv_addr(uint32_t buf, int r, int c) {
  return buf + r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
}

template <bool kKV8>
__global__ void __launch_bounds__(DecLayout<kKV8>::kThreads, 1)
    decode_attn_kernel(const __grid_constant__ CUtensorMap map_kp,
                       const __grid_constant__ CUtensorMap map_vp, DecAttnArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  using Lay = DecLayout<kKV8>;
  constexpr int kDecStages = Lay::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(smem);
  const uint32_t bars = base + Lay::kBar;
  auto full = [&](int s) { return bars + kDecBarFull + 8 * s; };
  auto empty = [&](int s) { return bars + kDecBarEmpty + 8 * s; };
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + Lay::kBar + kDecAbort);
  float* mlx = reinterpret_cast<float*>(smem + Lay::kML);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u0 = blockIdx.x * a.per_cta, u1 = min(a.units, u0 + a.per_cta);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&map_kp);
      tma_prefetch_map(&map_vp);
      int p = 0;
      for (int u = u0; u < u1; ++u) {
        const UnitInfo x = unit_info(a, u, true);
        if (!x.valid) continue;
        const int st = p % kDecStages;
        if (*abort_flag || !mbar_wait(empty(st), ((p / kDecStages) & 1) ^ 1, a.wait_ns)) {
          report_status(a.status, kStatusTimeout);
          *abort_flag = 1;
          break;
        }
        const uint32_t sb = base + st * Lay::kStage;
        const int row0 = (x.page * a.G + x.g) * kBlock;
        mbar_arrive_expect_tx(full(st), Lay::kStage);
        if (kKV8) {  // one 128 x 128-byte box per tile
          tma_load_2d(sb, &map_kp, full(st), 0, row0);
          tma_load_2d(sb + Lay::kTile, &map_vp, full(st), 0, row0);
        } else {     // two 64-element panels per tile
          tma_load_2d(sb, &map_kp, full(st), 0, row0);
          tma_load_2d(sb + kPanel, &map_kp, full(st), 64, row0);
          tma_load_2d(sb + Lay::kTile, &map_vp, full(st), 0, row0);
          tma_load_2d(sb + Lay::kTile + kPanel, &map_vp, full(st), 64, row0);
        }
        ++p;
      }
      if (*abort_flag) {  // in-flight loads land before the producer exits (default limit)
        for (int x = (p > kDecStages ? p - kDecStages : 0); x < p; ++x)
          mbar_wait(full(x % kDecStages), (x / kDecStages) & 1, kDefaultWaitNs);
      }
    }
    return;  // the producer takes no part in the compute warps' named barriers
  }

  // ---------------- compute warps 1..8: group gr takes the staged units p with p % 2 == gr ----
  const int gr = (warp - 1) >> 2, w = (warp - 1) & 3;
  const uint32_t bar_id = 1 + gr;  // the group's named barrier
  const int gid = lane >> 2, tq = lane & 3;
  const uint32_t vp = base + Lay::kPriv + (gr * 4 + w) * Lay::kPrivWarp;  // e4m3 only
  uint32_t qa[8][4];
  int cur_sg = -1;
  int p = -1;  // staged units seen so far, minus one
  const float ninf = -__int_as_float(0x7f800000);
  for (int u = u0; u < u1; ++u) {
    const UnitInfo x = unit_info(a, u, false);
    if (!x.valid) {
      if (gr == 0 && w == 0 && lane < kHeads)
        a.plse[static_cast<size_t>(u) * kHeads + lane] = ninf;
      continue;
    }
    if (++p % Lay::kGroups != gr) continue;  // another group's unit
    const int sg = x.s * a.G + x.g;
    if (sg != cur_sg) {  // query fragments of this (sequence, group), straight from global
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(a.q + static_cast<size_t>(sg) *
                                                                        kHeads * kDim);
      if (kKV8) {
        // fp16, with k elements 2tq, 2tq+1, 2tq+8, 2tq+9 of each k-step taken from dimensions
        // 4tq .. 4tq+3 (the K fragments below use the same permutation)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qa[kk][0] = bf16x2_to_f16x2(q32[(gid * kDim + kk * 16 + tq * 4) >> 1]);
          qa[kk][1] = bf16x2_to_f16x2(q32[((gid + 8) * kDim + kk * 16 + tq * 4) >> 1]);
          qa[kk][2] = bf16x2_to_f16x2(q32[(gid * kDim + kk * 16 + tq * 4 + 2) >> 1]);
          qa[kk][3] = bf16x2_to_f16x2(q32[((gid + 8) * kDim + kk * 16 + tq * 4 + 2) >> 1]);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qa[kk][0] = q32[(gid * kDim + kk * 16 + tq * 2) >> 1];
          qa[kk][1] = q32[((gid + 8) * kDim + kk * 16 + tq * 2) >> 1];
          qa[kk][2] = q32[(gid * kDim + kk * 16 + 8 + tq * 2) >> 1];
          qa[kk][3] = q32[((gid + 8) * kDim + kk * 16 + 8 + tq * 2) >> 1];
        }
      }
      cur_sg = sg;
    }
    const int st = p % kDecStages;
    // The stage's previous unit (p - kDecStages) is this group's own previous unit when there
    // are as many stages as groups; with more stages it would belong to another group, whose
    // release must be waited for (as the producer does before refilling the stage) so that the
    // full barrier is at most one phase ahead of this wait: a group skips the other groups' units,
    // and a parity test on a barrier two phases behind would pass on the stale phase.
    bool ok = !*abort_flag &&
              (p < kDecStages ||
               mbar_wait(empty(st), ((p / kDecStages) & 1) ^ 1, a.wait_ns)) &&
              mbar_wait(full(st), (p / kDecStages) & 1, a.wait_ns);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) report_status(a.status, kStatusTimeout);
      *abort_flag = 1;  // keep going with whatever is in the buffer: every warp still meets
                        // the same barriers, and the status word marks the output invalid
    }
    const uint32_t kt = base + st * Lay::kStage, vt = kt + Lay::kTile;
    if (kKV8) {
      // V columns [32w, 32w+32) of all 128 keys: 4 keys per step, 8 lanes per key
#pragma unroll 4
      for (int it = 0; it < 32; ++it) {
        const int r = it * 4 + (lane >> 3);
        const int c = 2 * w + ((lane & 7) >> 2);
        const uint32_t src = vt + r * 128 + ((c ^ (r & 7)) << 4) + (lane & 3) * 4;
        uint32_t h0, h1;
        e4m3x4_to_f16x4(ld_shared_u32(src), h0, h1);
        st_shared_v2(vpriv_addr(vp, r, (lane & 7) >> 1) + (lane & 1) * 8, h0, h1);
      }
      __syncwarp();
    }
    const int par = (p / Lay::kGroups) & 1;                // parity of the group's units
    const uint32_t pt = base + Lay::kP + (gr * 2 + par) * Lay::kPBytes;  // this unit's P tile
    float* mx = mlx + gr * (Lay::kMLGroup / 4) + par * (2 * 4 * kHeads);  // [4 warps][16] maxima
    float* ls = mx + 4 * kHeads;                                          // [4 warps][16] sums
    // S = q K^T over this warp's 32 keys: 4 n-tiles of 8 keys
    float sacc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[j][e] = 0.f;
      if (kKV8) {
        // B fragment of key w*32 + 8j + gid: bytes [4tq, 4tq + 4) of k-step kk's 16-byte chunk
        // (the 8 keys' rows hit 8 distinct chunks of the swizzle: no bank conflicts)
        const int kr = w * 32 + j * 8 + gid;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t b0, b1;
          e4m3x4_to_f16x4(ld_shared_u32(kt + kr * 128 + ((kk ^ (kr & 7)) << 4) + tq * 4), b0,
                          b1);
          mma_m16n8k16_f16(sacc[j], qa[kk], b0, b1);
        }
      } else {
        const int key = w * 32 + j * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
          uint32_t r[4];
          ldmatrix_x4(swz(kt, key, 2 * kk + (lane >> 3)), r);
          mma_m16n8k16_bf16(sacc[j], qa[kk], r[0], r[1]);
          mma_m16n8k16_bf16(sacc[j], qa[kk + 1], r[2], r[3]);
        }
      }
    }
    if (kKV8) {  // K and V of the stage have been read
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(st));
    }
    // scale, causal limit, this warp's row maxima (rows gid and gid+8) over its 32 keys
    float m0 = ninf, m1 = ninf;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = w * 32 + j * 8 + tq * 2 + (e & 1);
        const float z = key <= x.lim ? sacc[j][e] * a.scale_log2 : ninf;
        sacc[j][e] = z;
        if (e < 2) m0 = fmaxf(m0, z);
        else m1 = fmaxf(m1, z);
      }
    }
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
    if (tq == 0) {
      mx[w * kHeads + gid] = m0;
      mx[w * kHeads + gid + 8] = m1;
    }
    named_barrier(bar_id, 128);
    // row maxima over the page (key 0 is always in range, so they are finite)
    float M0 = mx[gid], M1 = mx[gid + 8];
#pragma unroll
    for (int q = 1; q < 4; ++q) {
      M0 = fmaxf(M0, mx[q * kHeads + gid]);
      M1 = fmaxf(M1, mx[q * kHeads + gid + 8]);
    }
    // P = exp2(z - M) for this warp's keys -> bf16 (fp16 with an e4m3 cache) into the shared P
    // tile; partial row sums
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float p0 = exp2f(sacc[j][0] - M0), p1 = exp2f(sacc[j][1] - M0);
      const float p2 = exp2f(sacc[j][2] - M1), p3 = exp2f(sacc[j][3] - M1);
      l0 += p0 + p1;
      l1 += p2 + p3;
      const int chunk = w * 4 + j;  // keys [8 chunk, 8 chunk + 8)
      st_shared_u32(dec_p_addr(pt, gid, chunk) + tq * 4,
                    kKV8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1));
      st_shared_u32(dec_p_addr(pt, gid + 8, chunk) + tq * 4,
                    kKV8 ? pack_f16x2(p2, p3) : pack_bf16x2(p2, p3));
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (tq == 0) {
      ls[w * kHeads + gid] = l0;
      ls[w * kHeads + gid + 8] = l1;
    }
    named_barrier(bar_id, 128);
    const float L0 = ls[gid] + ls[kHeads + gid] + ls[2 * kHeads + gid] + ls[3 * kHeads + gid];
    const float L1 = ls[gid + 8] + ls[kHeads + gid + 8] + ls[2 * kHeads + gid + 8] +
                     ls[3 * kHeads + gid + 8];
    // O[:, 32w, 32w + 32) = P V over all 128 keys: 8 k-steps x 4 n-tiles of 8 dims
    float oacc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[nt][e] = 0.f;
    const int mtx = lane >> 3;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t pa[4];
      ldmatrix_x4(dec_p_addr(pt, lane & 15, 2 * kk + (lane >> 4)), pa);
      const int key = kk * 16 + (mtx & 1) * 8 + (lane & 7);
#pragma unroll
      for (int nt = 0; nt < 4; nt += 2) {
        uint32_t r[4];
        if (kKV8) {
          ldmatrix_x4_trans(vpriv_addr(vp, key, nt + (mtx >> 1)), r);
          mma_m16n8k16_f16(oacc[nt], pa, r[0], r[1]);
          mma_m16n8k16_f16(oacc[nt + 1], pa, r[2], r[3]);
        } else {
          ldmatrix_x4_trans(swz(vt, key, w * 4 + nt + (mtx >> 1)), r);
          mma_m16n8k16_bf16(oacc[nt], pa, r[0], r[1]);
          mma_m16n8k16_bf16(oacc[nt + 1], pa, r[2], r[3]);
        }
      }
    }
    __syncwarp();
    if (!kKV8 && lane == 0) mbar_arrive(empty(st));
    const float i0 = 1.f / L0, i1 = 1.f / L1;
    float* dst = a.po + static_cast<size_t>(u) * kHeads * kDim;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int d = (w * 4 + nt) * 8 + tq * 2;
      *reinterpret_cast<float2*>(dst + gid * kDim + d) =
          make_float2(oacc[nt][0] * i0, oacc[nt][1] * i0);
      *reinterpret_cast<float2*>(dst + (gid + 8) * kDim + d) =
          make_float2(oacc[nt][2] * i1, oacc[nt][3] * i1);
    }
    if (w == 0 && tq == 0) {
      const float ln2 = 0.6931471805599453f;
      a.plse[static_cast<size_t>(u) * kHeads + gid] = (M0 + __log2f(L0)) * ln2;
      a.plse[static_cast<size_t>(u) * kHeads + gid + 8] = (M1 + __log2f(L1)) * ln2;
    }
  }
}

// Combine of the k slot partials of each (sequence, head): fixed slot order, no atomics.
struct DecCombineArgs {
  const float* po;
  const float* plse;
  int32_t batch, G, k;
  __nv_bfloat16* o;  // [batch][G*16][128]
  float* lse;        // [G*16][batch]
};

__global__ void __launch_bounds__(128) decode_combine_kernel(DecCombineArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  const int s = blockIdx.x, g = blockIdx.y, t = threadIdx.x, hh = t >> 3, d0 = (t & 7) * 16;
  const size_t u0 = (static_cast<size_t>(s) * a.G + g) * a.k;
  float M = -__int_as_float(0x7f800000);
  for (int j = 0; j < a.k; ++j) M = fmaxf(M, a.plse[(u0 + j) * kHeads + hh]);
  float acc[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) acc[q] = 0.f;
  float den = 0.f;
#pragma unroll 4
  for (int j = 0; j < a.k; ++j) {
    const float l = a.plse[(u0 + j) * kHeads + hh];
    if (l == -__int_as_float(0x7f800000)) continue;
    const float wgt = __expf(l - M);
    den += wgt;
    const float4* src = reinterpret_cast<const float4*>(a.po + ((u0 + j) * kHeads + hh) * kDim + d0);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 x = src[c];
      acc[4 * c] += wgt * x.x;
      acc[4 * c + 1] += wgt * x.y;
      acc[4 * c + 2] += wgt * x.z;
      acc[4 * c + 3] += wgt * x.w;
    }
  }
  const float inv = 1.f / den;
  const int h = g * kHeads + hh;
  uint4* dst = reinterpret_cast<uint4*>(a.o + (static_cast<size_t>(s) * a.G * kHeads + h) * kDim + d0);
#pragma unroll
  for (int c = 0; c < 2; ++c)
    dst[c] = make_uint4(pack_bf16x2(acc[8 * c] * inv, acc[8 * c + 1] * inv),
                        pack_bf16x2(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv),
                        pack_bf16x2(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv),
                        pack_bf16x2(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv));
  if ((t & 7) == 0) a.lse[static_cast<size_t>(h) * a.batch + s] = M + __logf(den);
}

}  // namespace

size_t decode_select_workspace_bytes(int batch, int G, int max_pages) {
  return static_cast<size_t>(batch) * G * max_pages * sizeof(float4);
}

cudaError_t launch_decode_select(const CUtensorMap& map_k, const CUtensorMap& map_q,
                                 const int32_t* page_table, const int32_t* seq_lens, int batch,
                                 int max_pages, int num_pages, int G, int k, bool fp8,
                                 float* scores, int32_t* sel, float* sel_score,
                                 float* block_scores, int32_t* status, uint64_t wait_ns,
                                 int num_sms, cudaStream_t stream, int kb0, int kb1,
                                 float* cand_score, int32_t* cand_block) {
  ScanArgs a{};
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.G = G;
  a.kb0 = kb0;
  a.kb1 = kb1;
  a.scores = reinterpret_cast<float4*>(scores);
  a.status = status;
  a.wait_ns = wait_ns;
  const int grid = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(fp8 ? scan_ctas_per_sm<true>()
                                                                     : scan_ctas_per_sm<false>()) *
                                                 num_sms,
                                             static_cast<int64_t>(batch) * max_pages)));
  cudaError_t e;
  if (fp8) {
    if ((e = cudaFuncSetAttribute(decode_scan_kernel<true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  scan_smem<true>())) != cudaSuccess)
      return e;
    if ((e = launch_pdl(decode_scan_kernel<true>, dim3(grid), dim3(kScanThreads),
                        scan_smem<true>(), stream, map_k, map_q, a)) != cudaSuccess)
      return e;
  } else {
    if ((e = cudaFuncSetAttribute(decode_scan_kernel<false>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  scan_smem<false>())) != cudaSuccess)
      return e;
    if ((e = launch_pdl(decode_scan_kernel<false>, dim3(grid), dim3(kScanThreads),
                        scan_smem<false>(), stream, map_k, map_q, a)) != cudaSuccess)
      return e;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  TopkArgs t{};
  t.scores = a.scores;
  t.seq_lens = seq_lens;
  t.batch = batch;
  t.max_pages = max_pages;
  t.G = G;
  t.k = k;
  t.kb0 = kb0;
  t.kb1 = kb1;
  t.sel = sel;
  t.sel_score = sel_score;
  t.block_scores = block_scores;
  t.cand_score = cand_score;
  t.cand_block = cand_block;
  t.status = status;
  return launch_pdl(decode_topk_kernel, dim3(batch * G), dim3(128), 0, stream, t);
}

size_t decode_attn_workspace_bytes(int batch, int G, int k) {
  const size_t units = static_cast<size_t>(batch) * G * k;
  return units * kHeads * kDim * sizeof(float) + units * kHeads * sizeof(float);
}

cudaError_t launch_decode_attn(const CUtensorMap& map_kp, const CUtensorMap& map_vp,
                               const void* q, const int32_t* sel, const int32_t* page_table,
                               const int32_t* seq_lens, int batch, int max_pages, int num_pages,
                               int G, int k, float scale, uint8_t* scratch, void* o, float* lse,
                               int32_t* status, uint64_t wait_ns, int num_sms,
                               cudaStream_t stream, bool kv_fp8) {
  DecAttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.sel = sel;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.G = G;
  a.k = k;
  a.units = batch * G * k;
  const int grid = std::max(1, std::min(num_sms, a.units));
  a.per_cta = (a.units + grid - 1) / grid;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.po = reinterpret_cast<float*>(scratch);
  a.plse = reinterpret_cast<float*>(scratch + static_cast<size_t>(a.units) * kHeads * kDim * 4);
  a.status = status;
  a.wait_ns = wait_ns;
  cudaError_t e;
  if (kv_fp8) {
    constexpr uint32_t smem = DecLayout<true>::kSmem;
    if ((e = cudaFuncSetAttribute(decode_attn_kernel<true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
      return e;
    if ((e = launch_pdl(decode_attn_kernel<true>, dim3(grid), dim3(DecLayout<true>::kThreads),
                        smem, stream, map_kp, map_vp, a)) != cudaSuccess)
      return e;
  } else {
    constexpr uint32_t smem = DecLayout<false>::kSmem;
    if ((e = cudaFuncSetAttribute(decode_attn_kernel<false>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
      return e;
    if ((e = launch_pdl(decode_attn_kernel<false>, dim3(grid), dim3(DecLayout<false>::kThreads),
                        smem, stream, map_kp, map_vp, a)) != cudaSuccess)
      return e;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  DecCombineArgs c{a.po, a.plse, batch, G, k, static_cast<__nv_bfloat16*>(o), lse};
  if ((e = launch_pdl(decode_combine_kernel, dim3(batch, G), dim3(128), 0, stream, c)) !=
      cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace msa
