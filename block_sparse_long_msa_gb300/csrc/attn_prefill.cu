// Main branch for prefill, KV-outer ("MiniMax M3 算力省 20 倍", section 四: the outer loop runs
// over KV blocks; the queries that selected a block are gathered into 128-row tensor-core tiles;
// hot blocks are pre-split along the query dimension over many CTAs; partial results are merged
// by a two-phase combine without atomics).  Exactness per section 二: softmax over exactly the
// selected tokens, causal inside the local block.
//
// Per query chunk [q0, q1) (chunks bound the partial-output workspace):
//   1. sched_hist   per (group, query block): which tokens chose which block (bitmask in shared
//                   memory), per-block counts -> hist[g][b][qb]
//   2. sched_scan   per (group, block): exclusive prefix of hist over query blocks, list length
//   3. sched_bases  one CTA: list offsets over (group, block), work-item offsets over
//                   (query range, group, block)
//   4. sched_items  per (query range, group, block): work items of at most kItemTokens tokens.
//                   Items are ordered query-range-major, so the CTAs working at any moment
//                   gather the queries of one range (a few tens of MB) and L2 serves the
//                   repeated gathers of each query for its k blocks.
//   5. sched_fill   per (group, query block): every (token, slot) lands at its place, lists stay
//                   in ascending token order (deterministic, no global atomics)
//   6. attn_kv_outer persistent tcgen05 kernel over work items, taken from a counter (below)
//   7. combine      per (token, group): fixed slot order, LSE-weighted merge
#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"

namespace msa {

namespace {

constexpr int kTileTokens = 8;                            // 8 tokens x 16 heads = 128 MMA rows
constexpr int kHeadsPerGroup = 16;
constexpr int kItemTiles = 16;                            // tiles sharing one K/V staging
constexpr int kItemTokens = kItemTiles * kTileTokens;     // 128
constexpr uint32_t kPanel = 16384;
constexpr int kMaxRanges = 32;                            // <= 32: one warp lane per range
constexpr int kRangeBlocks = 16;                          // query blocks per range (2,048 tokens)
constexpr int64_t kScanEntries = 65536;                   // bound on nr * G * nbk

// ------------------------------------------------------------------------------------------
// Scheduling
// ------------------------------------------------------------------------------------------
struct SchedArgs {
  const int32_t* sel;  // [G][L][k]
  int64_t L;
  int32_t G, k;
  int32_t q0;          // first query of the chunk (multiple of 128)
  int32_t nbq;         // query blocks in the chunk
  int32_t nbk;         // key blocks referenced by the chunk (= last query block + 1)
  int32_t rq, nr;      // query blocks per query range, number of ranges (<= kMaxRanges)
  int32_t* hist;       // [G][nbk][nbq]
  int32_t* cnt;        // [G*nbk]
  int32_t* list_base;  // [G*nbk]
  int32_t* rstart;     // [nr][G][nbk]: offset of the range's first token in the (g, b) list
  int32_t* rcnt;       // [nr][G][nbk]: tokens of the range in the (g, b) list
  int32_t* item_base;  // [nr][G][nbk]
  int32_t* n_items;    // [1]
  int4* items;         // {g, b, start, count}
  int32_t* list;       // (token << 4) | slot
  int32_t* pos;        // [(il*G + g)*k + s]: list position of the slot's unit, -1 if none
  int64_t units;       // capacity of list / pos: chunk * G * k
  int64_t max_items;   // capacity of items
  int32_t* status;
};

// Shared-memory bitmask of the (up to 128) tokens of query block qb that selected block b.
// Returns false (and flags the status word) for ids outside [0, qb].
__device__ __forceinline__ void build_block_mask(const SchedArgs& a, int g, int qb,
                                                 uint32_t* mask) {
  const int t = threadIdx.x;
  for (int w = t; w < (qb + 1) * 4; w += blockDim.x) mask[w] = 0;
  __syncthreads();
  const int64_t i = static_cast<int64_t>(qb) * kBlock + t;
  if (t < kBlock && i < a.L) {
    const int32_t* row = a.sel + (static_cast<size_t>(g) * a.L + i) * a.k;
    for (int s = 0; s < a.k; ++s) {
      const int32_t b = row[s];
      if (b < 0) continue;
      if (b > qb) {
        report_status(a.status, kStatusBounds);
        continue;
      }
      atomicOr(&mask[b * 4 + (t >> 5)], 1u << (t & 31));
    }
  }
  __syncthreads();
}

__global__ void sched_hist_kernel(SchedArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  extern __shared__ uint32_t mask[];
  const int qbl = blockIdx.x, g = blockIdx.y;
  const int qb = a.q0 / kBlock + qbl;
  build_block_mask(a, g, qb, mask);
  for (int b = threadIdx.x; b <= qb; b += blockDim.x) {
    const int c = __popc(mask[b * 4]) + __popc(mask[b * 4 + 1]) + __popc(mask[b * 4 + 2]) +
                  __popc(mask[b * 4 + 3]);
    a.hist[(static_cast<size_t>(g) * a.nbk + b) * a.nbq + qbl] = c;
  }
}

// One warp per (group, block): exclusive prefix over the query blocks that can choose b.
__global__ void sched_scan_kernel(SchedArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= a.G * a.nbk) return;
  const int b = warp % a.nbk;
  const int qb0 = a.q0 / kBlock;
  int32_t* h = a.hist + static_cast<size_t>(warp) * a.nbq;
  const int first = b > qb0 ? b - qb0 : 0;
  int run = 0;
  for (int base = first; base < a.nbq; base += 32) {
    const int q = base + lane;
    const int v = q < a.nbq ? h[q] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (q < a.nbq) h[q] = run + incl - v;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) a.cnt[warp] = run;
  __syncwarp();
  // where each query range starts in this (g, b) list; ranges before the first query block
  // that can choose b start at 0
  int start = run;
  if (lane < a.nr) {
    const int q = lane * a.rq;
    start = q < first ? 0 : h[q];
  }
  const int next = __shfl_down_sync(0xffffffffu, start, 1);
  const int cnt = lane < a.nr ? (lane + 1 < a.nr ? next : run) - start : 0;
  // Consecutive ranges are merged into segments of at least one full work item (a sparse list
  // would otherwise be cut into short items, each reloading K and V for a few tokens); a
  // segment's tokens are listed under its last range, so its items run with that range's.
  int seg_cnt = 0, seg_start = 0, acc = 0, open_at = 0;
  for (int r = 0; r < a.nr; ++r) {
    const int c = __shfl_sync(0xffffffffu, cnt, r);
    const int st = __shfl_sync(0xffffffffu, start, r);
    if (acc == 0) open_at = st;
    acc += c;
    if (acc >= kItemTokens || r == a.nr - 1) {
      if (lane == r) {
        seg_cnt = acc;
        seg_start = open_at;
      }
      acc = 0;
    }
  }
  if (lane < a.nr) {
    const size_t idx = static_cast<size_t>(lane) * a.G * a.nbk + warp;
    a.rstart[idx] = seg_start;
    a.rcnt[idx] = seg_cnt;
  }
}

__device__ __forceinline__ int items_of(int c) {
  return (c + kItemTokens - 1) / kItemTokens;
}

// Exclusive scan of n values (val(i)) by one CTA of 1024 threads into out; returns the total.
template <typename F>
__device__ int block_exclusive_scan(int n, F val, int32_t* out, int32_t* warp_sums,
                                    int32_t* carry) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  if (t == 0) *carry = 0;
  __syncthreads();
  for (int base = 0; base < n; base += 1024) {
    const int idx = base + t;
    const int v = idx < n ? val(idx) : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
      const int s = warp_sums[lane];
      int x = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      warp_sums[lane] = x - s;
    }
    __syncthreads();
    if (idx < n) out[idx] = *carry + warp_sums[w] + incl - v;
    __syncthreads();
    if (t == 1023) *carry += warp_sums[w] + incl;
    __syncthreads();
  }
  return *carry;
}

// One CTA: list offsets over (group, block), item offsets over (range, group, block).
__global__ void __launch_bounds__(1024) sched_bases_kernel(SchedArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  const int32_t* cnt = a.cnt;
  const int32_t* rcnt = a.rcnt;
  block_exclusive_scan(a.G * a.nbk, [cnt](int i) { return cnt[i]; }, a.list_base, warp_sums,
                       &carry);
  const int total = block_exclusive_scan(
      a.nr * a.G * a.nbk, [rcnt](int i) { return items_of(rcnt[i]); }, a.item_base, warp_sums,
      &carry);
  if (threadIdx.x == 0) {
    *a.n_items = total;
    a.n_items[1] = 0;  // the attention kernel's work counter
  }
}

__global__ void sched_items_kernel(SchedArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.nr * a.G * a.nbk) return;
  const int gb = idx % (a.G * a.nbk);
  const int g = gb / a.nbk, b = gb % a.nbk;
  const int c = a.rcnt[idx], base = a.list_base[gb] + a.rstart[idx], ib = a.item_base[idx];
  for (int q = 0; q * kItemTokens < c; ++q) {
    if (!MSA_IN_RANGE(a.status, kSiteSchedItem, ib + q, a.max_items, idx)) break;
    a.items[ib + q] = make_int4(g, b, base + q * kItemTokens, min(kItemTokens, c - q * kItemTokens));
  }
}

__global__ void sched_fill_kernel(SchedArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  extern __shared__ uint32_t mask[];
  const int qbl = blockIdx.x, g = blockIdx.y;
  const int qb = a.q0 / kBlock + qbl;
  build_block_mask(a, g, qb, mask);
  const int t = threadIdx.x;
  const int64_t i = static_cast<int64_t>(qb) * kBlock + t;
  if (t >= kBlock || i >= a.L) return;
  const int32_t* row = a.sel + (static_cast<size_t>(g) * a.L + i) * a.k;
  const int w = t >> 5;
  const uint32_t below = (1u << (t & 31)) - 1u;
  const size_t u0 = (static_cast<size_t>(qbl) * kBlock + t) * a.G * a.k + static_cast<size_t>(g) * a.k;
  for (int s = 0; s < a.k; ++s) {
    const int32_t b = row[s];
    if (b < 0 || b > qb) {
      a.pos[u0 + s] = -1;
      continue;
    }
    int rank = __popc(mask[b * 4 + w] & below);
    for (int q = 0; q < w; ++q) rank += __popc(mask[b * 4 + q]);
    const int gb = g * a.nbk + b;
    const int pos = a.list_base[gb] + a.hist[static_cast<size_t>(gb) * a.nbq + qbl] + rank;
    if (!MSA_IN_RANGE(a.status, kSiteSchedList, pos, a.units, i)) {
      a.pos[u0 + s] = -1;
      continue;
    }
    a.list[pos] = static_cast<int32_t>((i << 4) | s);
    a.pos[u0 + s] = pos;
  }
}

// ------------------------------------------------------------------------------------------
// KV-outer attention.  One persistent CTA per SM takes work items from a global counter as it
// has room for the next one (items of uneven size then even out across SMs; taken in order,
// they keep the query-range order that L2 relies on); per item it stages K_b
// and V_b of group g (TMA; V converted to fp16 in place) and the item's token list, then for
// every tile of 8 tokens gathers their 16 query heads (TMA, 16 rows per token) and runs
//   S = Q K^T (tcgen05, fp32 in TMEM) -> softmax rows (causal limit only in the local block)
//   -> P (fp16, written back into the same TMEM columns) -> O = P V (tcgen05, A from TMEM)
//   -> unnormalised partial O (fp16, staged and stored with TMA) + row max m and log-sum-exp.
// Roles (16 warps): 0 query-gather producer + token-list staging, 1 S = QK^T issuer, 2 K loader
// + O = PV issuer, 3 V loader + fp16 converter, 4-7 softmax of even tiles, 8-11 softmax of odd
// tiles, 12-15 epilogue.
// TMEM: columns [0,384) three S/P slots (tile T uses slot T % 3), [384,512) the O accumulator.
// The two MMA chains of a tile come from two threads: a commit covers only its own thread's
// MMAs, so each chain signals its consumer when it is done while the tensor pipe interleaves
// them.  K and V are single-buffered (K paced by the S issuer, V by the P.V issuer), which frees
// shared memory for a three-deep query ring that covers the gather latency.  Partial outputs
// are kept in work-list order, so a full tile leaves with two TMA stores, from one of two
// staging tiles.  The kernel's DRAM traffic is mostly these partial writes (4 KiB per (token,
// group, block) unit).
// ------------------------------------------------------------------------------------------
struct AttnArgs {
  const int4* items;
  const int32_t* n_items;
  int32_t* next_item;     // work counter: each CTA takes the next item when it has room
  const int32_t* list;
  int32_t G, k, q0;
  int32_t q1, nbk;        // end of the chunk's queries, key blocks the chunk can select
  int64_t units, max_items;  // capacities of list / partials and of items
  float scale_log2;       // softmax scale * log2(e)
  __half* po;             // [list position][16][128] unnormalised partial O (fp16)
  float* pm;              // [list position][16] row max (natural-log units)
  float* plse;            // same, log-sum-exp
  int32_t* status;
  uint64_t wait_ns;
};

struct ItemMeta {
  int32_t g, b, count, start;  // start: list position of the item's first token
  int32_t tok[kItemTokens];  // (token << 4) | slot
};

constexpr int kQStages = 3;
constexpr int kMetaRing = 4;  // > items that can be in flight between the gather and the epilogue
constexpr uint32_t kSmemK = 0;                             // K of the current item (32 KB)
constexpr uint32_t kSmemV = 32768;                         // V of the current item (32 KB)
constexpr uint32_t kSmemQ = 65536;                         // 3 x 32 KB
constexpr uint32_t kSmemO = kSmemQ + kQStages * 32768;     // 2 x O staging tile (TMA stores)
constexpr uint32_t kSmemMeta = kSmemO + 2 * 32768;         // 4 x ItemMeta
constexpr uint32_t kSmemBar = kSmemMeta + kMetaRing * sizeof(ItemMeta);
constexpr uint32_t kAttnBarBytes = 512;
// the dynamic shared memory must start on a 1024-byte boundary (checked at kernel entry): the
// layout uses all but a few hundred bytes of the 227 KB a CTA may have
constexpr uint32_t kAttnSmem = kSmemBar + kAttnBarBytes;
static_assert(kAttnSmem <= 232448, "attention kernel shared memory");
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_f16_f32(128, 128, false, true);  // P, V in fp16

// barrier block offsets (bytes from kSmemBar)
constexpr uint32_t kBMetaFull = 0;     // [4]
constexpr uint32_t kBMetaEmpty = 32;   // [4]
constexpr uint32_t kBKFull = 64, kBKEmpty = 72, kBVFull = 80, kBVEmpty = 88, kBVReady = 96;
constexpr uint32_t kBQFull = 104;      // [3]
constexpr uint32_t kBQEmpty = 128;     // [3]
constexpr uint32_t kBSFull = 152;      // [6]: slot * 2 + softmax warpgroup
constexpr uint32_t kBPFull = 200;      // [6]
constexpr uint32_t kBSPFree = 248;     // [3]
constexpr uint32_t kBOFull = 272, kBOEmpty = 280, kBDrain = 288;
constexpr uint32_t kTmemSlot = 296, kAbort = 300;
static_assert(kBQFull + 8 * kQStages <= kBQEmpty && kBQEmpty + 8 * kQStages <= kBSFull, "bars");
static_assert(kBSFull + 48 <= kBPFull && kBPFull + 48 <= kBSPFree && kBSPFree + 24 <= kBOFull,
              "bars");
static_assert(kAbort + 4 <= kAttnBarBytes, "bars");

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

__global__ void __launch_bounds__(512, 1)
    attn_kv_outer_kernel(const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v,
                         const __grid_constant__ CUtensorMap map_po,
                         const __grid_constant__ CUtensorMap map_po_tok, AttnArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const uint32_t base = smem_u32(smem);
  if (base & 1023u) {  // the swizzled tiles need 1024-byte alignment; never seen, but checked
    if (threadIdx.x == 0) report_status(a.status, kStatusBounds);
    return;
  }
  const uint32_t bars = base + kSmemBar;
  auto meta_full = [&](int r) { return bars + kBMetaFull + 8 * r; };
  auto meta_empty = [&](int r) { return bars + kBMetaEmpty + 8 * r; };
  const uint32_t k_full = bars + kBKFull, k_empty = bars + kBKEmpty;
  const uint32_t v_full = bars + kBVFull, v_empty = bars + kBVEmpty, v_ready = bars + kBVReady;
  auto q_full = [&](int s) { return bars + kBQFull + 8 * s; };
  auto q_empty = [&](int s) { return bars + kBQEmpty + 8 * s; };
  auto s_full = [&](int sw) { return bars + kBSFull + 8 * sw; };
  auto p_full = [&](int sw) { return bars + kBPFull + 8 * sw; };
  auto sp_free = [&](int s) { return bars + kBSPFree + 8 * s; };
  const uint32_t o_full = bars + kBOFull, o_empty = bars + kBOEmpty;
  const uint32_t drain_bar = bars + kBDrain;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kSmemBar + kTmemSlot);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + kSmemBar + kAbort);
  ItemMeta* meta = reinterpret_cast<ItemMeta*>(smem + kSmemMeta);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n_items = *a.n_items;
  if (!MSA_IN_RANGE(a.status, kSiteSchedItem, n_items, a.max_items + 1, -1))
    n_items = static_cast<int>(a.max_items);

  if (threadIdx.x == 0) {
    for (int r = 0; r < kMetaRing; ++r) {
      mbar_init(meta_full(r), 1);
      // the epilogue's 128 threads when the item is finished, and one arrival from each of the
      // eight softmax warps once it has copied the item's fields (a warpgroup may own no tile of
      // an item, and nothing else would keep the slot from being refilled under its reads)
      mbar_init(meta_empty(r), 128 + 8);
    }
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(v_ready, 32);
    for (int q = 0; q < kQStages; ++q) {
      mbar_init(q_full(q), 1);
      mbar_init(q_empty(q), 1);
    }
    for (int sw = 0; sw < 6; ++sw) {
      mbar_init(s_full(sw), 1);
      mbar_init(p_full(sw), 128);
    }
    for (int q = 0; q < 3; ++q) mbar_init(sp_free(q), 1);
    mbar_init(o_full, 1);
    mbar_init(o_empty, 128);
    mbar_init(drain_bar, 2);  // one commit from each MMA issuer
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
    // --------------------- token lists + query gathers ---------------------
    int T = 0, q_issued = 0;
    bool ok = true;
    if (lane == 0) tma_prefetch_map(&map_q);
    for (int n = 0; ok; ++n) {
      const int r = n % kMetaRing;
      if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(meta_empty(r),
                                                             ((n / kMetaRing) & 1) ^ 1,
                                                             a.wait_ns))) {
        ok = false;
        break;
      }
      int it = 0;
      if (lane == 0) it = atomicAdd(a.next_item, 1);
      it = __shfl_sync(0xffffffffu, it, 0);
      ItemMeta& m = meta[r];
      if (it >= n_items) {  // no work left: an end marker for the other roles
        if (lane == 0) {
          m.count = -1;
          mbar_arrive(meta_full(r));
        }
        break;
      }
      int4 item = a.items[it];
      // checked build: a malformed item or token is clamped into range (the status word then
      // marks the results invalid) so that every role still sees a consistent item
      if (!MSA_IN_RANGE(a.status, kSiteAttnItem, item.x, a.G, it)) item.x = 0;
      if (!MSA_IN_RANGE(a.status, kSiteAttnItem, item.y, a.nbk, it)) item.y = 0;
      if (!MSA_IN_RANGE(a.status, kSiteAttnItem, item.w - 1, kItemTokens, it)) item.w = 1;
      if (!MSA_IN_RANGE(a.status, kSiteAttnItem, item.z, a.units - item.w + 1, it)) item.z = 0;
      for (int j = lane; j < item.w; j += 32) {
        int32_t e = a.list[item.z + j];
        // a token of the chunk, at or after the first token of the item's block; a slot < k
        const int lo = max(a.q0, item.y * kBlock);
        if (!MSA_IN_RANGE(a.status, kSiteAttnToken, (e >> 4) - lo, a.q1 - lo, it) ||
            !MSA_IN_RANGE(a.status, kSiteAttnToken, e & 15, a.k, it))
          e = lo << 4;
        m.tok[j] = e;
      }
      if (lane == 0) {
        m.g = item.x;
        m.b = item.y;
        m.count = item.w;
        m.start = item.z;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(meta_full(r));
      for (int t0 = 0; t0 < item.w; t0 += kTileTokens, ++T) {
        const int qs = T % kQStages;
        if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(q_empty(qs),
                                                               ((T / kQStages) & 1) ^ 1,
                                                               a.wait_ns))) {
          ok = false;
          break;
        }
        const int nt = min(kTileTokens, item.w - t0);
        const uint32_t qb = base + kSmemQ + qs * 32768u;
        if (lane == 0) mbar_arrive_expect_tx(q_full(qs), nt * 4096);
        __syncwarp();
        if (lane < 2 * nt) {  // lanes 0..2n-1: token lane/2, 64-column half lane%2
          const int tk = lane >> 1, half = lane & 1;
          const int i = m.tok[t0 + tk] >> 4;
          tma_load_3d(qb + half * kPanel + tk * 2048, &map_q, q_full(qs), half * 64,
                      item.x * kHeadsPerGroup, i);
        }
        ++q_issued;
      }
    }
    if (!ok) {
      if (lane == 0) report_status(a.status, kStatusTimeout);
      *abort_flag = 1;
      if (lane == 0)  // let in-flight gathers land before the CTA can exit
        for (int x = (q_issued > kQStages ? q_issued - kQStages : 0); x < q_issued; ++x)
          mbar_wait(q_full(x % kQStages), (x / kQStages) & 1, kDefaultWaitNs);
    }
  } else if (warp == 1) {
    // ---------------------------- S = Q K^T issuer ----------------------------
    // S and P.V are issued by two threads (this one and lane 0 of warp 2).  A tcgen05.commit
    // covers only the MMAs of the thread that issues it, so each chain signals its consumer as
    // soon as it is done while the tensor pipe interleaves the two threads' independent chains.
    if (lane == 0) {
      bool ok = true;
      int T = 0;
      for (int n = 0; ok; ++n) {
        const int r = n % kMetaRing;
        if (*abort_flag || !mbar_wait(meta_full(r), (n / kMetaRing) & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        const int cnt = meta[r].count;
        if (cnt < 0) break;
        if (!mbar_wait(k_full, n & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        for (int t0 = 0; t0 < cnt; t0 += kTileTokens, ++T) {
          const int qs = T % kQStages, s3 = T % 3;
          // S(T) reuses the S/P slot of tile T-3: in-order issue keeps the parities unambiguous
          if (*abort_flag || !mbar_wait(q_full(qs), (T / kQStages) & 1, a.wait_ns) ||
              !mbar_wait(sp_free(s3), ((T / 3) & 1) ^ 1, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + s3 * 128;
          const uint32_t qb = base + kSmemQ + qs * 32768u, kb = base + kSmemK;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
            mma_bf16_ss(d, sdesc_sw128(qb + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                        kIdescQK, kk > 0);
          }
          mma_commit(s_full(s3 * 2 + (T & 1)));
          mma_commit(q_empty(qs));
        }
        if (!ok) break;
        mma_commit(k_empty);  // the item's last S: K may be replaced once these are done
      }
      if (!ok) {
        report_status(a.status, kStatusTimeout);
        *abort_flag = 1;
      }
      mma_commit(drain_bar);
      mbar_wait(drain_bar, 0, kDefaultWaitNs);
    }
  } else if (warp == 2) {
    // --------------------- K loader + O = P V issuer (polling) ---------------------
    if (lane == 0) {
      tma_prefetch_map(&map_k);
      int n_mine = 0x7fffffff;  // items of this CTA, known at the end marker
      int nk = 0;                        // items whose K has been requested
      int b_n = 0, b_cnt = -1, b_t0 = 0, b_T = 0;  // P.V cursor
      bool ok = true, idle = false;
      uint64_t idle_since = 0;
      while (ok && (nk < n_mine || b_n < n_mine)) {
        bool progressed = false;
        // one test of the item's barrier decides both cases: the end marker, or a K to load
        if (nk < n_mine && mbar_test_wait(meta_full(nk % kMetaRing), (nk / kMetaRing) & 1)) {
          const int r = nk % kMetaRing;
          if (meta[r].count < 0) {
            n_mine = nk;
            progressed = true;
          } else if (mbar_test_wait(k_empty, (nk & 1) ^ 1)) {
            const int g = meta[r].g, b = meta[r].b;
            mbar_arrive_expect_tx(k_full, 32768);
            tma_load_3d(base + kSmemK, &map_k, k_full, 0, g, b * kBlock);
            tma_load_3d(base + kSmemK + kPanel, &map_k, k_full, 64, g, b * kBlock);
            ++nk;
            progressed = true;
          }
        }
        if (b_n < n_mine) {
          if (b_cnt < 0 && mbar_test_wait(v_ready, b_n & 1)) {  // V of item b_n converted
            b_cnt = meta[b_n % kMetaRing].count;
            b_t0 = 0;
          }
          const int s3 = b_T % 3;
          if (b_cnt >= 0 && mbar_test_wait(p_full(s3 * 2 + (b_T & 1)), (b_T / 6) & 1) &&
              mbar_test_wait(o_empty, (b_T & 1) ^ 1)) {
            tc_fence_after();
            const uint32_t pa = tmem + s3 * 128, vb = base + kSmemV;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ts(tmem + 384, pa + kk * 8, sdesc_sw128(vb + kk * 2048, kPanel, 1024),
                         kIdescPV, kk > 0);
            mma_commit(o_full);
            mma_commit(sp_free(s3));
            ++b_T;
            b_t0 += kTileTokens;
            if (b_t0 >= b_cnt) {  // the item's last P.V: V may be replaced once it is done
              mma_commit(v_empty);
              ++b_n;
              b_cnt = -1;
            }
            progressed = true;
          }
        }
        if (progressed) {
          idle = false;
        } else {
          const uint64_t now = globaltimer_ns();
          if (!idle) {
            idle = true;
            idle_since = now;
          } else if (now - idle_since > a.wait_ns || *abort_flag) {
            ok = false;
          }
        }
      }
      if (!ok) {
        report_status(a.status, kStatusTimeout);
        *abort_flag = 1;
        if (nk > 0) mbar_wait(k_full, (nk - 1) & 1, kDefaultWaitNs);
      }
      mma_commit(drain_bar);
      mbar_wait(drain_bar, 0, kDefaultWaitNs);
    }
  } else if (warp == 3) {
    // ------------- V loader + converter: bf16 -> fp16 in place -------------
    // Exact for N(0,1)-range values (bf16 carries 8 significant bits, fp16 11); lets P be
    // rounded to fp16 instead of bf16 for the P.V product.
    if (lane == 0) tma_prefetch_map(&map_v);
    int issued = 0;
    bool ok = true;
    for (int n = 0;; ++n) {
      const int r = n % kMetaRing;
      if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(meta_full(r), (n / kMetaRing) & 1,
                                                             a.wait_ns))) {
        ok = false;
        break;
      }
      if (meta[r].count < 0) break;
      if (!__all_sync(0xffffffffu, mbar_wait(v_empty, (n & 1) ^ 1, a.wait_ns))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        const int g = meta[r].g, b = meta[r].b;
        mbar_arrive_expect_tx(v_full, 32768);
        tma_load_3d(base + kSmemV, &map_v, v_full, 0, g, b * kBlock);
        tma_load_3d(base + kSmemV + kPanel, &map_v, v_full, 64, g, b * kBlock);
      }
      ++issued;
      if (!__all_sync(0xffffffffu, mbar_wait(v_full, n & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      const uint32_t vb = base + kSmemV;
#pragma unroll 4
      for (int c = lane; c < 2048; c += 32) {
        uint4 x = ld_shared_v4(vb + c * 16);
        x.x = bf16x2_to_f16x2(x.x);
        x.y = bf16x2_to_f16x2(x.y);
        x.z = bf16x2_to_f16x2(x.z);
        x.w = bf16x2_to_f16x2(x.w);
        st_shared_v4(vb + c * 16, x.x, x.y, x.z, x.w);
      }
      fence_proxy_async_smem();
      mbar_arrive(v_ready);
    }
    if (!ok) {
      if (lane == 0) report_status(a.status, kStatusTimeout);
      *abort_flag = 1;
      if (lane == 0 && issued > 0) mbar_wait(v_full, (issued - 1) & 1, kDefaultWaitNs);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------- softmax -------------------------------
    const int wg = (warp - 4) >> 2;          // handles tiles with (T & 1) == wg
    const int row = (warp & 3) * 32 + lane;  // TMEM lane = MMA row
    const int tk = row >> 4, hh = row & 15;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int T = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int r = n % kMetaRing;
      if (!__all_sync(0xffffffffu, mbar_wait(meta_full(r), (n / kMetaRing) & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      const ItemMeta& m = meta[r];
      if (m.count < 0) break;
      // the slot is refilled only after every softmax warp has copied these fields (its arrival
      // below) and the epilogue has finished the item; the token ids of a tile are read before
      // the tile's P is released, so the item cannot be finished under those reads
      const int count = m.count, b = m.b, start = m.start;
      __syncwarp();
      if (lane == 0) mbar_arrive(meta_empty(r));
      for (int t0 = 0; t0 < count; t0 += kTileTokens, ++T) {
        if ((T & 1) != wg) continue;
        const int s3 = T % 3;
        const uint32_t sa = tmem + lane_base + s3 * 128;
        if (!__all_sync(0xffffffffu, mbar_wait(s_full(s3 * 2 + wg), (T / 6) & 1, a.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool valid = t0 + tk < count;
        const int i = valid ? m.tok[t0 + tk] >> 4 : 0;
        const int lim = valid ? min(i - b * kBlock, kBlock - 1) : kBlock - 1;
        // tiles of non-local tokens (all but the first 16 of a block's list) need no mask
        const bool unmasked = __all_sync(0xffffffffu, lim >= kBlock - 1);
        // pass 1: row max of the scaled logits (log2 units); two TMEM loads per wait
        float mraw = -__int_as_float(0x7f800000);
#pragma unroll 1
        for (int c = 0; c < 4; c += 2) {
          uint32_t v0[32], v1[32];
          tmem_ld32(sa + c * 32, v0);
          tmem_ld32(sa + c * 32 + 32, v1);
          tmem_ld_wait();
          if (unmasked) {
            float m4[4] = {mraw, mraw, mraw, mraw};  // four independent three-input chains
#pragma unroll
            for (int q = 0; q < 32; ++q)
              m4[q & 3] = fmax3(m4[q & 3], __uint_as_float(v0[q]), __uint_as_float(v1[q]));
            mraw = fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              if (c * 32 + q <= lim) mraw = fmaxf(mraw, __uint_as_float(v0[q]));
              if (c * 32 + 32 + q <= lim) mraw = fmaxf(mraw, __uint_as_float(v1[q]));
            }
          }
        }
        const float m2 = mraw * a.scale_log2;  // the scale is positive
        // pass 2: p = exp2(s * scale - m2) -> fp16 pairs; keys [16c, 16c+16) go to columns
        // [8c, 8c+8), which hold S values this thread has already read
        float2 l2 = make_float2(0.f, 0.f);
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nm2 = make_float2(-m2, -m2);
#pragma unroll 1
        for (int c = 0; c < 8; c += 2) {
          uint32_t v[32], pk[16];
          tmem_ld16(sa + c * 16, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
          tmem_ld16(sa + c * 16 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 32; q += 2) {
            float2 t = ffma2(make_float2(__uint_as_float(v[q]), __uint_as_float(v[q + 1])), sc2,
                             nm2);
            float p0 = fast_exp2(t.x), p1 = fast_exp2(t.y);
            if (!unmasked) {
              const int j = c * 16 + q;
              p0 = j <= lim ? p0 : 0.f;
              p1 = j + 1 <= lim ? p1 : 0.f;
            }
            l2.x += p0;
            l2.y += p1;
            pk[q >> 1] = pack_f16x2(p0, p1);
          }
          tmem_st16(sa + c * 8, pk);
        }
        const float l = l2.x + l2.y;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full(s3 * 2 + wg));
        if (valid) {
          const size_t p = static_cast<size_t>(start) + t0 + tk;  // list position
          const float ln2 = 0.6931471805599453f;
          a.pm[p * kHeadsPerGroup + hh] = m2 * ln2;
          a.plse[p * kHeadsPerGroup + hh] = (m2 + __log2f(l)) * ln2;
        }
      }
    }
    if (!ok) {
      report_status(a.status, kStatusTimeout);
      *abort_flag = 1;
    }
  } else {
    // ------------------------------- epilogue -------------------------------
    // O (fp32, TMEM) -> fp16 rows in a 128-byte-swizzled staging tile (two, used alternately)
    // -> TMA stores: each token's 16 heads are 4 KB contiguous in the partial buffer, and the
    // tokens of a tile are consecutive list positions, so a full tile is two stores (one per
    // 64-column half) and a short last tile one store per (token, half).  Every epilogue thread
    // runs the same loop, so the named barriers always pair up; after an abort the waits are
    // skipped and nothing more is stored.
    const int et = threadIdx.x - 384;
    const int row = (warp & 3) * 32 + lane;
    if (et == 0) {
      tma_prefetch_map(&map_po);
      tma_prefetch_map(&map_po_tok);
    }
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int T = 0;
    for (int n = 0;; ++n) {
      const int r = n % kMetaRing;
      const bool okm = !*abort_flag && mbar_wait(meta_full(r), (n / kMetaRing) & 1, a.wait_ns);
      if (!__all_sync(0xffffffffu, okm)) {
        report_status(a.status, kStatusTimeout);
        *abort_flag = 1;
        break;
      }
      const ItemMeta& m = meta[r];
      if (m.count < 0) break;
      const int count = min(max(m.count, 0), kItemTokens);
      for (int t0 = 0; t0 < count; t0 += kTileTokens, ++T) {
        const bool oko = !*abort_flag && mbar_wait(o_full, T & 1, a.wait_ns);
        if (!__all_sync(0xffffffffu, oko)) {
          report_status(a.status, kStatusTimeout);
          *abort_flag = 1;
        }
        tc_fence_after();
        // O -> registers as fp16 pairs; the accumulator is released before the staging tile is
        // waited for, so the next P.V does not wait on the previous tile's TMA stores
        uint32_t ph[64];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v0[32], v1[32];
          tmem_ld32(tmem + lane_base + 384 + h * 64, v0);
          tmem_ld32(tmem + lane_base + 384 + h * 64 + 32, v1);
          tmem_ld_wait();
          if (h == 1) {  // the accumulator is in registers: the next P.V may start
            tc_fence_before();
            mbar_arrive(o_empty);
          }
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            ph[h * 32 + q] = pack_f16x2(__uint_as_float(v0[2 * q]), __uint_as_float(v0[2 * q + 1]));
            ph[h * 32 + 16 + q] =
                pack_f16x2(__uint_as_float(v1[2 * q]), __uint_as_float(v1[2 * q + 1]));
          }
        }
        // two staging tiles: this tile's was last used two tiles ago, whose stores have read it
        // once at most one (the previous tile's) bulk group is still reading
        const uint32_t stg = base + kSmemO + (T & 1) * 32768u;
        if (et < 16) bulk_wait_read1();
        named_barrier(1, 128);
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8)  // 16-byte chunk c8 = columns [8 c8, 8 c8 + 8)
          st_shared_v4(stg + sw128_offset(row, c8 * 8, 128), ph[4 * c8], ph[4 * c8 + 1],
                       ph[4 * c8 + 2], ph[4 * c8 + 3]);
        fence_proxy_async_smem();
        named_barrier(1, 128);
        // Partials are kept in list order, so a full tile's 8 tokens x 16 heads are 128
        // consecutive rows: two TMA stores (one per 64-column half).  A short last tile stores
        // token by token (rows past it belong to the next item).
        if (et < 16) {
          const bool full = t0 + kTileTokens <= count;
          const int tk = full ? 0 : et >> 1, h = full ? et : et & 1;
          if (!*abort_flag && (full ? et < 2 : t0 + tk < count))
            tma_store_2d(full ? &map_po : &map_po_tok, stg + h * kPanel + tk * 2048, h * 64,
                         (m.start + t0 + tk) * kHeadsPerGroup);
          bulk_commit();
        }
      }
      mbar_arrive(meta_empty(r));
    }
    if (et < 16) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// Combine: per (token, group), 128 threads; thread t covers head t/8, dims (t%8)*16 .. +16.
//   M = max_s lse_s, den = sum_s exp(lse_s - M), o = sum_s exp(m_s - M) * O~_s / den,
//   lse = M + ln(den).  Slots in fixed ascending order; padding (-1) skipped.
// ------------------------------------------------------------------------------------------
struct CombineArgs {
  const int32_t* pos;          // [(il*G + g)*k + s]: list position of each slot, -1 if none
  const __half* po;
  const float* pm;
  const float* plse;
  int64_t L;                   // rows of sel / o / lse
  int32_t G, k, q0, nrows;     // rows q0 .. q0+nrows-1
  __nv_bfloat16* o;            // [L][G*16][128]
  float* lse;                  // [G*16][L]
  int64_t units;               // capacity of the partials
  int32_t* status;
};

__global__ void __launch_bounds__(128) combine_kernel(CombineArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  const int il = blockIdx.x, g = blockIdx.y;
  const int64_t i = static_cast<int64_t>(a.q0) + il;
  const int t = threadIdx.x, hh = t >> 3, d0 = (t & 7) * 16;
  const int32_t* prow = a.pos + (static_cast<size_t>(il) * a.G + g) * a.k;
  // a slot's list position: -1 (padding, or an id that was flagged) or below units; the checked
  // build treats a position past the partials as padding
  auto slot_pos = [&](int s) {
    const int32_t p = prow[s];
    return p >= 0 && MSA_IN_RANGE(a.status, kSiteCombinePos, p, a.units, i * a.G + g) ? p : -1;
  };
  float M = -__int_as_float(0x7f800000);
  for (int s = 0; s < a.k; ++s) {
    const int32_t p = slot_pos(s);
    if (p >= 0) M = fmaxf(M, a.plse[static_cast<size_t>(p) * kHeadsPerGroup + hh]);
  }
  float acc[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) acc[q] = 0.f;
  float den = 0.f;
  // unrolled by four so that several slots' partial loads are in flight per thread (the order of
  // the sums is unchanged)
#pragma unroll 4
  for (int s = 0; s < a.k; ++s) {
    const int32_t p = slot_pos(s);
    if (p < 0) continue;  // padding (and out-of-range ids, which were flagged)
    const size_t r = static_cast<size_t>(p) * kHeadsPerGroup + hh;
    den += __expf(a.plse[r] - M);
    const float w = __expf(a.pm[r] - M);
    const uint4* src = reinterpret_cast<const uint4*>(a.po + r * kDim + d0);
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const uint4 x = src[h2];
      const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wd[q]));
        acc[h2 * 8 + 2 * q] += w * f.x;
        acc[h2 * 8 + 2 * q + 1] += w * f.y;
      }
    }
  }
  const float inv = 1.f / den;
  const int h = g * kHeadsPerGroup + hh;
  uint4* dst = reinterpret_cast<uint4*>(a.o + (static_cast<size_t>(i) * a.G * kHeadsPerGroup + h) * kDim + d0);
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    uint4 w;
    w.x = pack_bf16x2(acc[h2 * 8 + 0] * inv, acc[h2 * 8 + 1] * inv);
    w.y = pack_bf16x2(acc[h2 * 8 + 2] * inv, acc[h2 * 8 + 3] * inv);
    w.z = pack_bf16x2(acc[h2 * 8 + 4] * inv, acc[h2 * 8 + 5] * inv);
    w.w = pack_bf16x2(acc[h2 * 8 + 6] * inv, acc[h2 * 8 + 7] * inv);
    dst[h2] = w;
  }
  if ((t & 7) == 0) a.lse[static_cast<size_t>(h) * a.L + i] = M + __logf(den);
}

}  // namespace

// Query ranges of a chunk: 2,048 tokens each (16 query blocks; at most kMaxRanges, so longer
// chunks get longer ranges).  Work items run range by range, so the query gathers of the CTAs
// working at one time fall in one range (32 MiB of q at 64 heads), which L2 holds; each list is
// cut at range boundaries only where it has a full item's worth of tokens (sched_scan).
RangePlan plan_ranges(int64_t q0, int64_t q1, int G) {
  RangePlan p{};
  const int64_t nbq = (q1 - q0 + kBlock - 1) / kBlock, nbk = (q1 + kBlock - 1) / kBlock;
  int64_t nr_want = std::min<int64_t>(kMaxRanges, (nbq + kRangeBlocks - 1) / kRangeBlocks);
  // the one-CTA scan of sched_bases walks nr * G * nbk item counts: keep it to 64 rounds
  nr_want = std::max<int64_t>(1, std::min<int64_t>(nr_want, kScanEntries / (G * nbk)));
  p.rq = static_cast<int>((nbq + nr_want - 1) / nr_want);
  p.nr = static_cast<int>((nbq + p.rq - 1) / p.rq);
  return p;
}

// five scheduling kernels, the attention kernel, the combine
int prefill_chunk_launches() { return 7; }

PrefillWorkspace prefill_workspace_layout(int64_t L, int G, int k, int64_t chunk) {
  PrefillWorkspace w{};
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const int64_t nbk = (L + kBlock - 1) / kBlock;
  const int64_t nbq = (chunk + kBlock - 1) / kBlock;
  const int64_t units = chunk * G * k;
  // ranges a chunk of nbq query blocks can have (at most; plan_ranges)
  const int64_t nr = std::min<int64_t>(kMaxRanges, (nbq + kRangeBlocks - 1) / kRangeBlocks);
  const int64_t max_items = nr * G * nbk + (units + kItemTokens - 1) / kItemTokens;
  size_t off = 256;  // status header
  w.hist = off;      off += up(sizeof(int32_t) * G * nbk * nbq);
  w.cnt = off;       off += up(sizeof(int32_t) * G * nbk);
  w.list_base = off; off += up(sizeof(int32_t) * G * nbk);
  w.rstart = off;    off += up(sizeof(int32_t) * nr * G * nbk);
  w.rcnt = off;      off += up(sizeof(int32_t) * nr * G * nbk);
  w.item_base = off; off += up(sizeof(int32_t) * nr * G * nbk);
  w.n_items = off;   off += 256;
  w.items = off;     off += up(sizeof(int4) * max_items);
  w.list = off;      off += up(sizeof(int32_t) * units);
  w.pos = off;       off += up(sizeof(int32_t) * units);
  w.pm = off;        off += up(sizeof(float) * units * kHeadsPerGroup);
  w.plse = off;      off += up(sizeof(float) * units * kHeadsPerGroup);
  w.po = off;        off += up(sizeof(__half) * units * kHeadsPerGroup * kDim);
  w.total = off;
  w.chunk = chunk;
  w.max_items = max_items;
  return w;
}

cudaError_t launch_attn_prefill_chunk(const CUtensorMap& map_q, const CUtensorMap& map_k,
                                      const CUtensorMap& map_v, const int32_t* sel, int64_t L,
                                      int G, int k, float scale, int64_t q0, int64_t q1,
                                      uint8_t* ws, const PrefillWorkspace& w, void* o, float* lse,
                                      uint64_t wait_ns, int num_sms, cudaStream_t stream,
                                      cudaEvent_t* marks) {
  SchedArgs s{};
  s.sel = sel;
  s.L = L;
  s.G = G;
  s.k = k;
  s.q0 = static_cast<int32_t>(q0);
  s.nbq = static_cast<int32_t>((q1 - q0 + kBlock - 1) / kBlock);
  s.nbk = static_cast<int32_t>((q1 + kBlock - 1) / kBlock);
  s.hist = reinterpret_cast<int32_t*>(ws + w.hist);
  s.cnt = reinterpret_cast<int32_t*>(ws + w.cnt);
  s.list_base = reinterpret_cast<int32_t*>(ws + w.list_base);
  s.item_base = reinterpret_cast<int32_t*>(ws + w.item_base);
  s.rstart = reinterpret_cast<int32_t*>(ws + w.rstart);
  s.rcnt = reinterpret_cast<int32_t*>(ws + w.rcnt);
  const RangePlan plan = plan_ranges(q0, q1, G);
  s.rq = plan.rq;
  s.nr = plan.nr;
  s.n_items = reinterpret_cast<int32_t*>(ws + w.n_items);
  s.items = reinterpret_cast<int4*>(ws + w.items);
  s.list = reinterpret_cast<int32_t*>(ws + w.list);
  s.pos = reinterpret_cast<int32_t*>(ws + w.pos);
  s.units = w.chunk * G * k;
  s.max_items = w.max_items;
  s.status = reinterpret_cast<int32_t*>(ws);
  const size_t mask_smem = static_cast<size_t>(s.nbk) * 16;
  cudaError_t e;
  if (mask_smem > 48 * 1024) {
    if ((e = cudaFuncSetAttribute(sched_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(mask_smem))) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(sched_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(mask_smem))) != cudaSuccess)
      return e;
  }
  const dim3 qgrid(s.nbq, G);
  if (marks && marks[0]) cudaEventRecord(marks[0], stream);
  const int pairs = G * s.nbk;
  if ((e = launch_pdl(sched_hist_kernel, qgrid, dim3(kBlock), mask_smem, stream, s)) !=
          cudaSuccess ||
      (e = launch_pdl(sched_scan_kernel, dim3((pairs * 32 + 255) / 256), dim3(256), 0, stream,
                      s)) != cudaSuccess ||
      (e = launch_pdl(sched_bases_kernel, dim3(1), dim3(1024), 0, stream, s)) != cudaSuccess ||
      (e = launch_pdl(sched_items_kernel, dim3((s.nr * pairs + 255) / 256), dim3(256), 0, stream,
                      s)) != cudaSuccess ||
      (e = launch_pdl(sched_fill_kernel, qgrid, dim3(kBlock), mask_smem, stream, s)) !=
          cudaSuccess)
    return e;

  AttnArgs a{};
  a.items = s.items;
  a.n_items = s.n_items;
  a.next_item = s.n_items + 1;
  a.list = s.list;
  a.G = G;
  a.k = k;
  a.q0 = s.q0;
  a.q1 = static_cast<int32_t>(q1);
  a.nbk = s.nbk;
  a.units = s.units;
  a.max_items = s.max_items;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.po = reinterpret_cast<__half*>(ws + w.po);
  a.pm = reinterpret_cast<float*>(ws + w.pm);
  a.plse = reinterpret_cast<float*>(ws + w.plse);
  a.status = s.status;
  a.wait_ns = wait_ns;
  if ((e = cudaFuncSetAttribute(attn_kv_outer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kAttnSmem)) != cudaSuccess)
    return e;
  // partial O as a 2-D fp16 tensor [positions * 16 rows][128]: the epilogue's TMA stores, a
  // full tile (128 rows) or one token (16 rows) at a time
  CUtensorMap map_po, map_po_tok;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(kDim),
                              static_cast<uint64_t>(w.chunk) * G * k * kHeadsPerGroup};
    const uint64_t strides[1] = {kDim * 2};
    const uint32_t box[2] = {64, kTileTokens * kHeadsPerGroup};
    const uint32_t box_tok[2] = {64, kHeadsPerGroup};
    if (!encode_tmap(&map_po, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.po, 2, dims, strides, box) ||
        !encode_tmap(&map_po_tok, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.po, 2, dims, strides,
                     box_tok))
      return cudaErrorInvalidValue;
  }
  const int grid = static_cast<int>(std::min<int64_t>(w.max_items, num_sms));
  if (marks && marks[1]) cudaEventRecord(marks[1], stream);
  if ((e = launch_pdl(attn_kv_outer_kernel, dim3(grid), dim3(512), kAttnSmem, stream, map_q,
                      map_k, map_v, map_po, map_po_tok, a)) != cudaSuccess)
    return e;

  CombineArgs c{};
  c.pos = s.pos;
  c.po = a.po;
  c.pm = a.pm;
  c.plse = a.plse;
  c.L = L;
  c.G = G;
  c.k = k;
  c.q0 = s.q0;
  c.nrows = static_cast<int32_t>(q1 - q0);
  c.o = reinterpret_cast<__nv_bfloat16*>(o);
  c.lse = lse;
  c.units = s.units;
  c.status = s.status;
  if (marks && marks[2]) cudaEventRecord(marks[2], stream);
  return launch_pdl(combine_kernel, dim3(c.nrows, G), dim3(128), 0, stream, c);
}

}  // namespace msa
