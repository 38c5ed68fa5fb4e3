// Merge step of the context-parallel index branch ("MiniMax M3.1 Flash 开放权重与部署要点", section
// 权重能下载之后，为什么还要先看 vLLM: the indexer's decode runs context-parallel over several
// GPUs).  Each shard of the key blocks has ranked its own blocks and kept its top-(k-1)
// (msa_index_candidates); every block of the global top-(k-1) is within the top-(k-1) of its own
// shard (fewer than k-1 blocks outrank it anywhere), so ranking the union of the shards'
// candidates by the same rule, (score desc, block asc), gives the selection of the whole range
// exactly ("MiniMax M3 算力省 20 倍", section 二: per-group top-k plus the forced local block).
#include "common.cuh"
#include "launch.h"

namespace msa {

namespace {

struct MergeArgs {
  const float* cand_score;    // [R][G][T][k-1]
  const int32_t* cand_block;  // [R][G][T][k-1]
  int32_t R, G, k;
  int64_t T;
  const int32_t* seq_lens;    // decode: [T]; nullptr: prefill (query t at position t)
  int32_t* sel;               // [G][T][k]
  float* sel_score;           // optional
  int32_t* status;
};

// One thread per (group, query) row: a register top-(k-1) over the R x (k-1) candidates.
__global__ void __launch_bounds__(128) index_merge_kernel(MergeArgs a) {
  pdl_enter();  // before any global memory access (launch_pdl)
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= a.G * a.T) return;
  const int g = static_cast<int>(r / a.T);
  const int64_t t = r % a.T;
  int32_t* out = a.sel + static_cast<size_t>(r) * a.k;
  float* out_s = a.sel_score ? a.sel_score + static_cast<size_t>(r) * a.k : nullptr;
  int32_t bi;
  if (a.seq_lens) {
    const int n = a.seq_lens[t];
    if (n <= 0) {
      report_status(a.status, kStatusBounds);
      for (int c = 0; c < a.k; ++c) {
        out[c] = -1;
        if (out_s) out_s[c] = -__int_as_float(0x7f800000);
      }
      return;
    }
    bi = (n - 1) / kBlock;
  } else {
    bi = static_cast<int32_t>(t / kBlock);
  }
  const int w = a.k - 1;
  TopList list;
  list.clear();
  int found = 0;
  for (int sh = 0; sh < a.R; ++sh) {
    const size_t off = ((static_cast<size_t>(sh) * a.G + g) * a.T + t) * w;
    for (int c = 0; c < w; ++c) {
      const int32_t b = a.cand_block[off + c];
      const bool beyond = b >= bi;  // not strictly before the query's own block
      if (beyond) report_status(a.status, kStatusBounds);
      const bool take = b >= 0 && !beyond;  // b < 0: padding
      // every thread of the warp inserts (an empty entry when there is nothing to take), so
      // the list's warp vote sees the whole warp
      list.insert(take ? a.cand_score[off + c] : -__int_as_float(0x7f800000),
                  take ? b : 0x7fffffff);
      found += take;
    }
  }
  const int n = min(min(w, bi), found);
  list.truncate_and_sort_by_block(n);
  write_sel_row(list, n, bi, a.k, out, out_s);
}

}  // namespace

cudaError_t launch_index_merge(const float* cand_score, const int32_t* cand_block,
                               int num_shards, int64_t T, int G, int k,
                               const int32_t* seq_lens, int32_t* sel, float* sel_score,
                               int32_t* status, cudaStream_t stream) {
  MergeArgs a{cand_score, cand_block, num_shards, G, k, T, seq_lens, sel, sel_score, status};
  const int64_t rows = static_cast<int64_t>(G) * T;
  const unsigned grid = static_cast<unsigned>((rows + 127) / 128);
  return launch_pdl(index_merge_kernel, dim3(grid), dim3(128), 0, stream, a);
}

}  // namespace msa
