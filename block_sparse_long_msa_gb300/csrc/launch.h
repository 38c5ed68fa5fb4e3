// Internal launch entry points of the MSA kernels (host side, C++).  The public C ABI in
// include/msa.h validates arguments and builds tensor maps, then calls these.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace msa {

// Launch with programmatic stream serialization: the kernel may begin while the previous kernel
// on the stream drains (its CTAs wait in pdl_enter, ptx.cuh, before touching global memory),
// which hides the launch latency between the back-to-back kernels of a call and between calls.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Keys per tile of the prefill index kernel (two blocks): the box height of its key tensor map.
constexpr int kIndexKeyTile = 256;
// fp8: index vectors are e4m3 (else bf16); the tensor maps' element type must match.
// block_scores (optional): [G][L][nb] pooled score of every block (+inf local, -inf later).
// kb0, kb1: the key blocks scored (0, nb for the selection); map_k starts at block kb0.  With
// cand_block set, each row's top-(k-1) of those blocks goes to cand_score / cand_block
// [G][L][k-1] in rank order instead of the selection (a context-parallel shard).
cudaError_t launch_index_select_prefill(const CUtensorMap& map_q, const CUtensorMap& map_k,
                                        int64_t L, int G, int k, bool fp8, int32_t* sel,
                                        float* sel_score, float* block_scores, int32_t* status,
                                        uint64_t wait_ns, cudaStream_t stream, int kb0 = 0,
                                        int kb1 = 0x7fffffff, float* cand_score = nullptr,
                                        int32_t* cand_block = nullptr);

// Byte offsets of the prefill main-branch workspace (after the 256-byte status header).
struct PrefillWorkspace {
  size_t hist, cnt, list_base, rstart, rcnt, item_base, n_items, items, list, pos, pm, plse, po,
      total;
  int64_t chunk, max_items;
};
PrefillWorkspace prefill_workspace_layout(int64_t L, int G, int k, int64_t chunk);
struct RangePlan {
  int rq, nr;  // query blocks per query range, number of ranges
};
RangePlan plan_ranges(int64_t q0, int64_t q1, int G);
// Kernel launches one call of launch_attn_prefill_chunk makes.
int prefill_chunk_launches();
cudaError_t launch_attn_prefill_chunk(const CUtensorMap& map_q, const CUtensorMap& map_k,
                                      const CUtensorMap& map_v, const int32_t* sel, int64_t L,
                                      int G, int k, float scale, int64_t q0, int64_t q1,
                                      uint8_t* ws, const PrefillWorkspace& w, void* o, float* lse,
                                      uint64_t wait_ns, int num_sms, cudaStream_t stream,
                                      cudaEvent_t* marks);

size_t decode_select_workspace_bytes(int batch, int G, int max_pages);
// kb0, kb1: the logical blocks scanned (0, max_pages for the selection).  With cand_block set,
// each (sequence, group) row's top-(k-1) of those blocks goes to cand_score / cand_block
// [G][batch][k-1] in rank order instead of the selection (a context-parallel shard).
cudaError_t launch_decode_select(const CUtensorMap& map_k, const CUtensorMap& map_q,
                                 const int32_t* page_table, const int32_t* seq_lens, int batch,
                                 int max_pages, int num_pages, int G, int k, bool fp8,
                                 float* scores, int32_t* sel, float* sel_score,
                                 float* block_scores, int32_t* status, uint64_t wait_ns,
                                 int num_sms, cudaStream_t stream, int kb0 = 0,
                                 int kb1 = 0x7fffffff, float* cand_score = nullptr,
                                 int32_t* cand_block = nullptr);
// Merge of the candidates of num_shards disjoint key-block shards ([R][G][T][k-1] each) into the
// selection sel [G][T][k] (sel_score optional): rank by (score desc, block asc), keep
// min(k-1, blocks before the query's own), add the local block, ascending, -1 padded.
// seq_lens: decode (query t at seq_lens[t]-1); nullptr: prefill (query t at position t).
cudaError_t launch_index_merge(const float* cand_score, const int32_t* cand_block,
                               int num_shards, int64_t T, int G, int k,
                               const int32_t* seq_lens, int32_t* sel, float* sel_score,
                               int32_t* status, cudaStream_t stream);
size_t decode_attn_workspace_bytes(int batch, int G, int k);
cudaError_t launch_decode_attn(const CUtensorMap& map_kp, const CUtensorMap& map_vp,
                               const void* q, const int32_t* sel, const int32_t* page_table,
                               const int32_t* seq_lens, int batch, int max_pages, int num_pages,
                               int G, int k, float scale, uint8_t* scratch, void* o, float* lse,
                               int32_t* status, uint64_t wait_ns, int num_sms,
                               cudaStream_t stream, bool kv_fp8 = false);

// Checked build (MSA_DEBUG_CHECKS): validation of the caller's index tensors, run before the
// kernels when debug_checks_enabled() (the environment variable MSA_DEBUG_CHECKS is set to a
// value other than "" or "0").  The release build compiles these to no-ops returning success.
bool debug_checks_enabled();
cudaError_t debug_check_prefill_sel(const int32_t* sel, int64_t L, int G, int k,
                                    int32_t* status, cudaStream_t stream);
cudaError_t debug_check_paged(const int32_t* page_table, const int32_t* seq_lens, int batch,
                              int max_pages, int num_pages, int32_t* status, cudaStream_t stream);
cudaError_t debug_check_decode_sel(const int32_t* sel, const int32_t* seq_lens, int batch, int G,
                                   int k, int max_pages, int32_t* status, cudaStream_t stream);

}  // namespace msa
