// Shared constants and small helpers of the MSA kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace msa {

constexpr int kBlock = 128;     // B: tokens per block / page
constexpr int kDim = 128;       // d = d_i
constexpr int kTopMax = 16;     // largest k supported
constexpr int kListMax = 15;    // non-local slots kept while scanning (k - 1 <= 15)

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s

// Checked build (compiled with MSA_DEBUG_CHECKS): the workspace header holds, next to the status
// word, a record of the first failed bounds check: int32 site at byte 16, then int64 value,
// bound and row at bytes 24, 32, 40 (msa_debug_record_t in include/msa.h).  Codes of the sites
// checked inside the kernels (msa_debug_site_t):
enum : int32_t {
  kSiteSchedList = 16,   // a (token, slot) list position past the chunk's units
  kSiteSchedItem = 17,   // a work item past the workspace's item capacity
  kSiteAttnItem = 18,    // a work item's group, block, token count or list range
  kSiteAttnToken = 19,   // a listed token outside the chunk or before the item's block
  kSiteCombinePos = 20,  // a slot's list position past the chunk's units
  kSiteDecodePage = 21,  // a scanned (sequence, logical page) outside [0, batch) x [0, max_pages)
  kSiteIndexRow = 22,    // a selection or candidate row past the query count
};

#if defined(MSA_DEBUG_CHECKS)
// Record a failed check (the first one wins) and flag MSA_ERR_DEVICE_BOUNDS; returns false so
// that the caller skips or clamps the access.
static __device__ __noinline__ bool debug_fail(int32_t* status, int32_t site, long long value,
                                               long long bound, long long row) {
  if (status) {
    if (atomicCAS(status + 4, 0, site) == 0) {
      long long* rec = reinterpret_cast<long long*>(status + 6);
      rec[0] = value;
      rec[1] = bound;
      rec[2] = row;
    }
    report_status(status, kStatusBounds);
  }
  return false;
}
// True when 0 <= value < bound; otherwise records the failure.  The release build compiles the
// check out entirely (the expression is the constant true and its operands are not evaluated).
#define MSA_IN_RANGE(status, site, value, bound, row)                                   \
  ((static_cast<long long>(value) >= 0 &&                                               \
    static_cast<long long>(value) < static_cast<long long>(bound)) ||                   \
   ::msa::debug_fail((status), (site), static_cast<long long>(value),                   \
                     static_cast<long long>(bound), static_cast<long long>(row)))
#else
#define MSA_IN_RANGE(status, site, value, bound, row) true
#endif

// (score desc, block asc): does (sa, ba) rank before (sb, bb)?
__device__ __forceinline__ bool ranks_before(float sa, int32_t ba, float sb, int32_t bb) {
  return sa > sb || (sa == sb && ba < bb);
}

// Register-resident top-kListMax list, kept sorted by rank.  Empty slots hold (-inf, INT_MAX).
struct TopList {
  float s[kListMax];
  int32_t b[kListMax];

  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int p = 0; p < kListMax; ++p) {
      s[p] = -__int_as_float(0x7f800000);
      b[p] = 0x7fffffff;
    }
  }
  // Insert (score, block) if it ranks before the current last entry.  Branch-free: walking from
  // the tail, entry p takes entry p-1 when the new pair ranks before p-1, the new pair when it
  // ranks before p only, and stays otherwise (the list is sorted, so these tests are monotone).
  // The warp skips the walk when none of its lanes has anything to insert.
  __device__ __forceinline__ void insert(float score, int32_t block) {
    const bool any = ranks_before(score, block, s[kListMax - 1], b[kListMax - 1]);
    if (!__any_sync(__activemask(), any)) return;
    bool c_here = any;  // the new pair ranks before entry p (p = kListMax - 1 first)
#pragma unroll
    for (int p = kListMax - 1; p > 0; --p) {
      const bool c_prev = ranks_before(score, block, s[p - 1], b[p - 1]);
      s[p] = c_prev ? s[p - 1] : (c_here ? score : s[p]);
      b[p] = c_prev ? b[p - 1] : (c_here ? block : b[p]);
      c_here = c_prev;
    }
    s[0] = c_here ? score : s[0];
    b[0] = c_here ? block : b[0];
  }
  // Keep the first `keep` entries (by rank), then sort them by ascending block id; entries past
  // `keep` become (-inf, INT_MAX) and sort to the end.
  __device__ __forceinline__ void truncate_and_sort_by_block(int keep) {
#pragma unroll
    for (int p = 0; p < kListMax; ++p)
      if (p >= keep) {
        s[p] = -__int_as_float(0x7f800000);
        b[p] = 0x7fffffff;
      }
    // odd-even transposition sort on block id
#pragma unroll
    for (int round = 0; round < kListMax; ++round) {
#pragma unroll
      for (int p = (round & 1); p + 1 < kListMax; p += 2) {
        if (b[p] > b[p + 1]) {
          const float ts = s[p];
          const int32_t tb = b[p];
          s[p] = s[p + 1];
          b[p] = b[p + 1];
          s[p + 1] = ts;
          b[p + 1] = tb;
        }
      }
    }
  }
};

// Write one selection row: the n non-local ids (ascending, in list.b[0..n)), then the local
// block, then -1 padding up to k.  Scores: pooled score, +inf for local, -inf for padding.
__device__ __forceinline__ void write_sel_row(const TopList& list, int n, int32_t local, int k,
                                              int32_t* sel_row, float* score_row) {
#pragma unroll
  for (int r = 0; r < kTopMax; ++r) {
    if (r >= k) break;
    int32_t id;
    float sc;
    if (r < n) {
      id = list.b[r < kListMax ? r : kListMax - 1];
      sc = list.s[r < kListMax ? r : kListMax - 1];
    } else if (r == n) {
      id = local;
      sc = __int_as_float(0x7f800000);
    } else {
      id = -1;
      sc = -__int_as_float(0x7f800000);
    }
    sel_row[r] = id;
    if (score_row) score_row[r] = sc;
  }
}

// Write one candidate row of a key-block shard (context-parallel index branch): the first n
// entries of the rank-ordered list (score desc, block asc), then (-inf, -1) up to width = k - 1.
__device__ __forceinline__ void write_cand_row(const TopList& list, int n, int width,
                                               float* score_row, int32_t* block_row) {
#pragma unroll
  for (int r = 0; r < kListMax; ++r) {
    if (r >= width) break;
    const bool real = r < n;
    score_row[r] = real ? list.s[r] : -__int_as_float(0x7f800000);
    block_row[r] = real ? list.b[r] : -1;
  }
}

}  // namespace msa
