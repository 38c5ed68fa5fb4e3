// Input validation of the checked build (compiled with MSA_DEBUG_CHECKS, switched on at run time
// by the environment variable MSA_DEBUG_CHECKS).  The release kernels already skip, and flag, an
// id that would address memory out of range; these kernels check the whole form the C ABI
// documents for the caller's index tensors, which the release path tolerates silently when it
// is memory-safe:
//   - a selection row ("MiniMax M3 算力省 20 倍", section 二 and section 三 item 4): ids
//     strictly ascending, each at most the query's own block, -1 only as trailing padding, and
//     the query's own block present;
//   - a paged sequence: 1 <= seq_lens[s] <= max_pages * 128, and every page-table entry of its
//     used logical pages in [0, num_pages).
// A failure is recorded in the workspace header (first one wins) next to MSA_ERR_DEVICE_BOUNDS.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace msa {

#if defined(MSA_DEBUG_CHECKS)

namespace {

// Input sites (msa_debug_site_t in include/msa.h).
enum : int32_t {
  kSiteSelRange = 1,
  kSiteSelOrder = 2,
  kSiteSelLocal = 3,
  kSiteSeqLen = 4,
  kSitePageId = 5,
};

// One selection row of width k for a query whose own block is bi; row_id names it in a record.
__device__ void check_sel_row(const int32_t* row, int k, int64_t bi, int64_t row_id,
                              int32_t* status) {
  int64_t prev = -1;
  bool pad = false;
  for (int j = 0; j < k; ++j) {
    const int32_t b = row[j];
    if (b == -1) {
      pad = true;
      continue;
    }
    if (b < 0 || b > bi) {
      debug_fail(status, kSiteSelRange, b, bi + 1, row_id);
      return;
    }
    if (pad || b <= prev) {
      debug_fail(status, kSiteSelOrder, j, k, row_id);
      return;
    }
    prev = b;
  }
  if (prev != bi) debug_fail(status, kSiteSelLocal, prev, bi + 1, row_id);
}

__global__ void check_prefill_sel_kernel(const int32_t* sel, int64_t L, int G, int k,
                                         int32_t* status) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= G * L) return;
  check_sel_row(sel + r * k, k, (r % L) / kBlock, r, status);
}

__global__ void check_paged_kernel(const int32_t* page_table, const int32_t* seq_lens, int batch,
                                   int max_pages, int num_pages, int32_t* status) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  const int64_t n = seq_lens[s];
  const int64_t n_max = static_cast<int64_t>(max_pages) * kBlock;
  if (n < 1 || n > n_max) {
    debug_fail(status, kSiteSeqLen, n, n_max + 1, s);
    return;
  }
  const int used = static_cast<int>((n + kBlock - 1) / kBlock);
  for (int p = 0; p < used; ++p) {
    const int32_t id = page_table[static_cast<int64_t>(s) * max_pages + p];
    if (id < 0 || id >= num_pages) {
      debug_fail(status, kSitePageId, id, num_pages, s);
      return;
    }
  }
}

// Rows of sequences with an invalid length are left to check_paged_kernel.
__global__ void check_decode_sel_kernel(const int32_t* sel, const int32_t* seq_lens, int batch,
                                        int G, int k, int max_pages, int32_t* status) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= static_cast<int64_t>(G) * batch) return;
  const int64_t n = seq_lens[r % batch];
  if (n < 1 || n > static_cast<int64_t>(max_pages) * kBlock) return;
  check_sel_row(sel + r * k, k, (n - 1) / kBlock, r, status);
}

unsigned blocks_for(int64_t n) { return static_cast<unsigned>((n + 255) / 256); }

}  // namespace

bool debug_checks_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("MSA_DEBUG_CHECKS");
    return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
  }();
  return on;
}

cudaError_t debug_check_prefill_sel(const int32_t* sel, int64_t L, int G, int k,
                                    int32_t* status, cudaStream_t stream) {
  if (L <= 0) return cudaSuccess;
  check_prefill_sel_kernel<<<blocks_for(G * L), 256, 0, stream>>>(sel, L, G, k, status);
  return cudaGetLastError();
}

cudaError_t debug_check_paged(const int32_t* page_table, const int32_t* seq_lens, int batch,
                              int max_pages, int num_pages, int32_t* status,
                              cudaStream_t stream) {
  if (batch <= 0) return cudaSuccess;
  check_paged_kernel<<<blocks_for(batch), 256, 0, stream>>>(page_table, seq_lens, batch,
                                                            max_pages, num_pages, status);
  return cudaGetLastError();
}

cudaError_t debug_check_decode_sel(const int32_t* sel, const int32_t* seq_lens, int batch, int G,
                                   int k, int max_pages, int32_t* status, cudaStream_t stream) {
  if (batch <= 0) return cudaSuccess;
  check_decode_sel_kernel<<<blocks_for(static_cast<int64_t>(G) * batch), 256, 0, stream>>>(
      sel, seq_lens, batch, G, k, max_pages, status);
  return cudaGetLastError();
}

#else  // release build: no input validation

bool debug_checks_enabled() { return false; }
cudaError_t debug_check_prefill_sel(const int32_t*, int64_t, int, int, int32_t*, cudaStream_t) {
  return cudaSuccess;
}
cudaError_t debug_check_paged(const int32_t*, const int32_t*, int, int, int, int32_t*,
                              cudaStream_t) {
  return cudaSuccess;
}
cudaError_t debug_check_decode_sel(const int32_t*, const int32_t*, int, int, int, int, int32_t*,
                                   cudaStream_t) {
  return cudaSuccess;
}

#endif

}  // namespace msa
