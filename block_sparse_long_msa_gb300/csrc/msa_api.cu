// C ABI of libmsa (declared in include/msa.h): argument checks, workspace carving, tensor-map
// encoding and kernel launches.  Nothing here allocates device memory or synchronizes, except
// msa_get_device_status, which reads the status word back.
#include "../../include/msa.h"
#include "common.cuh"
#include "launch.h"
#include "tmap.h"
#include "trace.h"

namespace {

using msa::kBlock;
using msa::kDim;

// bf16 tensor map with 128-byte swizzle; dims/strides innermost first (strides in bytes, one
// fewer than dims); box of 64 elements innermost.
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box) {
  return msa::encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides, box);
}

// Tensor map of index vectors (128 elements of the config's index type per row), 128-byte
// swizzle: dims[0] = 128 elements, strides in elements of the index type (converted to bytes
// here), box[0] = one 128-byte panel (64 bf16 or 128 e4m3 elements).
bool make_index_map(CUtensorMap* m, bool fp8, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_el, const uint32_t* box_rest) {
  const uint64_t esz = fp8 ? 1 : 2;
  uint64_t strides[3];
  uint32_t box[3];
  box[0] = fp8 ? 128 : 64;
  for (int r = 1; r < rank; ++r) {
    strides[r - 1] = strides_el[r - 1] * esz;
    box[r] = box_rest[r - 1];
  }
  return msa::encode_tmap(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          base, rank, dims, strides, box);
}

bool index_fp8(const msa_config_t* c) { return c->index_dtype == MSA_INDEX_E4M3; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

msa_status_t check_config(const msa_config_t* c) {
  if (!c) return MSA_ERR_INVALID_ARG;
  if (c->num_groups < 1 || c->heads_per_group < 1 || c->topk < 1 ||
      (c->index_dtype != MSA_INDEX_BF16 && c->index_dtype != MSA_INDEX_E4M3) ||
      c->wait_limit_ns < 0 || !(c->softmax_scale == c->softmax_scale))
    return MSA_ERR_INVALID_ARG;
  if (c->head_dim != kDim || c->index_dim != kDim || c->block_size != kBlock ||
      c->topk > msa::kTopMax)
    return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

uint64_t wait_ns(const msa_config_t* c) {
  return c->wait_limit_ns > 0 ? static_cast<uint64_t>(c->wait_limit_ns) : msa::kDefaultWaitNs;
}

int32_t* status_word(void* ws) { return reinterpret_cast<int32_t*>(ws); }

// Queries per prefill main-branch pass: bounds the partial-output workspace (G*k*16*128 bf16 per
// token, 256 KiB at G = 4, k = 16) to 16 GiB at most.
constexpr int64_t kPrefillChunk = 65536;
// The scheduler keeps a 16-byte token mask per key block in shared memory, and list entries
// pack the token index above a 4-bit slot.
constexpr int64_t kMaxPrefillTokens = 1536 * 1024;

int64_t prefill_chunk(int64_t L) {
  const int64_t rounded = (L + kBlock - 1) / kBlock * kBlock;
  return rounded < kPrefillChunk ? rounded : kPrefillChunk;
}

msa_status_t check_paged(const msa_paged_kv_t* p, bool need_kv) {
  if (!p || !p->k_idx_pool || !p->page_table || !p->seq_lens || p->batch < 0 ||
      p->max_pages < 1 || p->num_pages < 1 || !aligned16(p->k_idx_pool) ||
      (p->kv_dtype != MSA_KV_BF16 && p->kv_dtype != MSA_KV_E4M3))
    return MSA_ERR_INVALID_ARG;
  if (need_kv && (!p->k_pool || !p->v_pool || !aligned16(p->k_pool) || !aligned16(p->v_pool)))
    return MSA_ERR_INVALID_ARG;
  // page rows are addressed with 32-bit TMA coordinates
  if (static_cast<int64_t>(p->num_pages) * kBlock * 4 >= (static_cast<int64_t>(1) << 31))
    return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

bool sm_count(int* sms) {
  int dev = 0;
  return cudaGetDevice(&dev) == cudaSuccess &&
         cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
}

msa_status_t index_select_paged(const msa_config_t* cfg, const void* q_idx,
                                const msa_paged_kv_t* paged, int32_t* sel, float* sel_score,
                                float* block_scores, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  msa_status_t st = check_paged(paged, false);
  if (st != MSA_OK) return st;
  const int G = cfg->num_groups;
  if (G > 4) return MSA_ERR_UNSUPPORTED;
  if (ws_bytes < msa_index_select_workspace(cfg, paged->batch, 0, paged)) return MSA_ERR_WORKSPACE;
  if (paged->batch == 0) return MSA_OK;
  CUtensorMap mk, mq;
  const bool fp8 = index_fp8(cfg);
  {
    const uint64_t dims[2] = {kDim, static_cast<uint64_t>(paged->num_pages) * kBlock};
    const uint64_t strides[1] = {kDim};
    const uint32_t box[1] = {kBlock};
    if (!make_index_map(&mk, fp8, paged->k_idx_pool, 2, dims, strides, box)) return MSA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {kDim, static_cast<uint64_t>(paged->batch) * G};
    const uint64_t strides[1] = {kDim};
    const uint32_t box[1] = {static_cast<uint32_t>(G)};
    if (!make_index_map(&mq, fp8, q_idx, 2, dims, strides, box)) return MSA_ERR_CUDA;
  }
  int sms = 0;
  if (!sm_count(&sms)) return MSA_ERR_CUDA;
  if (msa::debug_checks_enabled() &&
      msa::debug_check_paged(paged->page_table, paged->seq_lens, paged->batch, paged->max_pages,
                             paged->num_pages, status_word(ws), stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  float* scores = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + MSA_WS_HEADER_BYTES);
  cudaError_t e = msa::launch_decode_select(mk, mq, paged->page_table, paged->seq_lens,
                                            paged->batch, paged->max_pages, paged->num_pages, G,
                                            cfg->topk, fp8, scores, sel, sel_score, block_scores,
                                            status_word(ws), wait_ns(cfg), sms, stream);
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* msa_status_string(msa_status_t s) {
  switch (s) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported size or configuration";
    case MSA_ERR_WORKSPACE: return "workspace too small";
    case MSA_ERR_CUDA: return "CUDA error";
    case MSA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MSA_ERR_DEVICE_BOUNDS: return "device index out of range";
  }
  return "unknown status";
}

// The status word and the checked build's record: bytes [0, 48) of the header.
constexpr size_t kStatusBytes = 48;

msa_status_t msa_reset_device_status(void* ws, cudaStream_t stream) {
  MSA_RANGE("msa_reset_device_status");
  if (!ws) return MSA_ERR_INVALID_ARG;
  return cudaMemsetAsync(ws, 0, kStatusBytes, stream) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

int32_t msa_debug_checks(void) {
#if defined(MSA_DEBUG_CHECKS)
  return 1 | (msa::debug_checks_enabled() ? 2 : 0);
#else
  return 0;
#endif
}

msa_status_t msa_get_debug_record(const void* ws, msa_debug_record_t* record,
                                  cudaStream_t stream) {
  MSA_RANGE("msa_get_debug_record");
  if (!ws || !record) return MSA_ERR_INVALID_ARG;
  *record = msa_debug_record_t{};
#if defined(MSA_DEBUG_CHECKS)
  static_assert(sizeof(msa_debug_record_t) == 32, "record layout");
  if (cudaMemcpyAsync(record, static_cast<const uint8_t*>(ws) + 16, sizeof *record,
                      cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
#else
  (void)stream;
  return MSA_ERR_UNSUPPORTED;
#endif
}

msa_status_t msa_get_device_status(const void* ws, cudaStream_t stream) {
  MSA_RANGE("msa_get_device_status");
  if (!ws) return MSA_ERR_INVALID_ARG;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (v == 0) return MSA_OK;
  if (v == MSA_ERR_DEVICE_TIMEOUT || v == MSA_ERR_DEVICE_BOUNDS) return static_cast<msa_status_t>(v);
  return MSA_ERR_CUDA;
}

size_t msa_index_select_workspace(const msa_config_t* cfg, int64_t num_queries, int64_t num_keys,
                                  const msa_paged_kv_t* paged) {
  (void)num_keys;
  if (check_config(cfg) != MSA_OK) return 0;
  size_t bytes = MSA_WS_HEADER_BYTES;
  if (paged) {
    if (num_queries < 0 || paged->max_pages < 0) return 0;
    // per-page pooled scores of the scan: [batch][G][max_pages] x 4 partial maxima
    bytes += align_up(msa::decode_select_workspace_bytes(static_cast<int>(num_queries),
                                                         cfg->num_groups, paged->max_pages),
                      256);
  }
  return bytes;
}

}  // extern "C"

namespace {

// Both index-branch entries: block_scores (optional) also receives every block's pooled score.
msa_status_t index_select(const msa_config_t* cfg, const void* q_idx, const void* k_idx,
                          int64_t L, const msa_paged_kv_t* paged, int32_t* sel, float* sel_score,
                          float* block_scores, void* ws, size_t ws_bytes, cudaStream_t stream) {
  msa_status_t st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!q_idx || !sel || !ws || !aligned16(q_idx)) return MSA_ERR_INVALID_ARG;
  const int G = cfg->num_groups;
  if (paged)
    return index_select_paged(cfg, q_idx, paged, sel, sel_score, block_scores, ws, ws_bytes,
                              stream);
  if (!k_idx || !aligned16(k_idx) || L < 0) return MSA_ERR_INVALID_ARG;
  if (G > 4) return MSA_ERR_UNSUPPORTED;  // odd G: one group per CTA
  if (L > (static_cast<int64_t>(1) << 31) - kBlock) return MSA_ERR_UNSUPPORTED;
  if (ws_bytes < msa_index_select_workspace(cfg, L, L, nullptr)) return MSA_ERR_WORKSPACE;
  if (L == 0) return MSA_OK;
  CUtensorMap mq, mk;
  const bool fp8 = index_fp8(cfg);
  {
    const uint64_t dims[3] = {kDim, static_cast<uint64_t>(G), static_cast<uint64_t>(L)};
    const uint64_t strides[2] = {kDim, static_cast<uint64_t>(G) * kDim};
    const uint32_t box[2] = {1, kBlock};
    if (!make_index_map(&mq, fp8, q_idx, 3, dims, strides, box)) return MSA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {kDim, static_cast<uint64_t>(L)};
    const uint64_t strides[1] = {kDim};
    const uint32_t box[1] = {msa::kIndexKeyTile};
    if (!make_index_map(&mk, fp8, k_idx, 2, dims, strides, box)) return MSA_ERR_CUDA;
  }
  cudaError_t e = msa::launch_index_select_prefill(mq, mk, L, G, cfg->topk, fp8, sel, sel_score,
                                                   block_scores, status_word(ws), wait_ns(cfg),
                                                   stream);
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // namespace

extern "C" {

msa_status_t msa_index_select(const msa_config_t* cfg, const void* q_idx, const void* k_idx,
                              int64_t L, const msa_paged_kv_t* paged, int32_t* sel,
                              float* sel_score, void* ws, size_t ws_bytes, cudaStream_t stream) {
  MSA_RANGE("msa_index_select");
  return index_select(cfg, q_idx, k_idx, L, paged, sel, sel_score, nullptr, ws, ws_bytes, stream);
}

msa_status_t msa_index_select_scores(const msa_config_t* cfg, const void* q_idx,
                                     const void* k_idx, int64_t L, const msa_paged_kv_t* paged,
                                     int32_t* sel, float* sel_score, float* block_scores,
                                     void* ws, size_t ws_bytes, cudaStream_t stream) {
  MSA_RANGE("msa_index_select_scores");
  if (!block_scores) return MSA_ERR_INVALID_ARG;
  return index_select(cfg, q_idx, k_idx, L, paged, sel, sel_score, block_scores, ws, ws_bytes,
                      stream);
}

msa_status_t msa_index_candidates(const msa_config_t* cfg, const void* q_idx, const void* k_idx,
                                  int64_t L, const msa_paged_kv_t* paged, int32_t block_begin,
                                  int32_t block_end, float* cand_score, int32_t* cand_block,
                                  void* ws, size_t ws_bytes, cudaStream_t stream) {
  MSA_RANGE("msa_index_candidates");
  msa_status_t st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!q_idx || !ws || !aligned16(q_idx) || block_begin < 0 || block_end < block_begin)
    return MSA_ERR_INVALID_ARG;
  const int G = cfg->num_groups;
  if (G > 4) return MSA_ERR_UNSUPPORTED;
  if (cfg->topk == 1) return MSA_OK;  // no candidate slots: the local block is the selection
  if (!cand_score || !cand_block) return MSA_ERR_INVALID_ARG;
  const bool fp8 = index_fp8(cfg);
  int sms = 0;
  if (paged) {
    if ((st = check_paged(paged, false)) != MSA_OK) return st;
    if (ws_bytes < msa_index_select_workspace(cfg, paged->batch, 0, paged))
      return MSA_ERR_WORKSPACE;
    if (paged->batch == 0) return MSA_OK;
    CUtensorMap mk, mq;
    {
      const uint64_t dims[2] = {kDim, static_cast<uint64_t>(paged->num_pages) * kBlock};
      const uint64_t strides[1] = {kDim};
      const uint32_t box[1] = {kBlock};
      if (!make_index_map(&mk, fp8, paged->k_idx_pool, 2, dims, strides, box))
        return MSA_ERR_CUDA;
    }
    {
      const uint64_t dims[2] = {kDim, static_cast<uint64_t>(paged->batch) * G};
      const uint64_t strides[1] = {kDim};
      const uint32_t box[1] = {static_cast<uint32_t>(G)};
      if (!make_index_map(&mq, fp8, q_idx, 2, dims, strides, box)) return MSA_ERR_CUDA;
    }
    if (!sm_count(&sms)) return MSA_ERR_CUDA;
    if (msa::debug_checks_enabled() &&
        msa::debug_check_paged(paged->page_table, paged->seq_lens, paged->batch,
                               paged->max_pages, paged->num_pages, status_word(ws),
                               stream) != cudaSuccess)
      return MSA_ERR_CUDA;
    const int kb1 = block_end < paged->max_pages ? block_end : paged->max_pages;
    float* scores = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + MSA_WS_HEADER_BYTES);
    cudaError_t e = msa::launch_decode_select(
        mk, mq, paged->page_table, paged->seq_lens, paged->batch, paged->max_pages,
        paged->num_pages, G, cfg->topk, fp8, scores, nullptr, nullptr, nullptr, status_word(ws),
        wait_ns(cfg), sms, stream, block_begin < kb1 ? block_begin : kb1, kb1, cand_score,
        cand_block);
    return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
  }
  if (!k_idx || !aligned16(k_idx) || L < 0) return MSA_ERR_INVALID_ARG;
  if (L > (static_cast<int64_t>(1) << 31) - kBlock) return MSA_ERR_UNSUPPORTED;
  if (ws_bytes < msa_index_select_workspace(cfg, L, L, nullptr)) return MSA_ERR_WORKSPACE;
  if (L == 0) return MSA_OK;
  const int64_t nb = (L + kBlock - 1) / kBlock;
  const int64_t kb1 = block_end < nb ? block_end : nb;
  const int64_t kb0 = block_begin < kb1 ? block_begin : kb1;
  // k_idx holds the keys of the shard only: positions [kb0 * B, min(kb1 * B, L))
  const int64_t rows = (kb1 * kBlock < L ? kb1 * kBlock : L) - kb0 * kBlock;
  CUtensorMap mq, mk;
  {
    const uint64_t dims[3] = {kDim, static_cast<uint64_t>(G), static_cast<uint64_t>(L)};
    const uint64_t strides[2] = {kDim, static_cast<uint64_t>(G) * kDim};
    const uint32_t box[2] = {1, kBlock};
    if (!make_index_map(&mq, fp8, q_idx, 3, dims, strides, box)) return MSA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {kDim, static_cast<uint64_t>(rows > 0 ? rows : 1)};
    const uint64_t strides[1] = {kDim};
    const uint32_t box[1] = {msa::kIndexKeyTile};
    if (!make_index_map(&mk, fp8, k_idx, 2, dims, strides, box)) return MSA_ERR_CUDA;
  }
  cudaError_t e = msa::launch_index_select_prefill(
      mq, mk, L, G, cfg->topk, fp8, nullptr, nullptr, nullptr, status_word(ws), wait_ns(cfg),
      stream, static_cast<int>(kb0), static_cast<int>(kb1), cand_score, cand_block);
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

msa_status_t msa_index_merge(const msa_config_t* cfg, int32_t num_shards,
                             const float* cand_score, const int32_t* cand_block, int64_t T,
                             const int32_t* seq_lens, int32_t* sel, float* sel_score, void* ws,
                             size_t ws_bytes, cudaStream_t stream) {
  MSA_RANGE("msa_index_merge");
  msa_status_t st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (num_shards < 1 || T < 0 || !sel || !ws) return MSA_ERR_INVALID_ARG;
  if (cfg->topk > 1 && (!cand_score || !cand_block)) return MSA_ERR_INVALID_ARG;
  if (ws_bytes < MSA_WS_HEADER_BYTES) return MSA_ERR_WORKSPACE;
  if (!seq_lens && T > (static_cast<int64_t>(1) << 31) - kBlock) return MSA_ERR_UNSUPPORTED;
  if (T == 0) return MSA_OK;
  cudaError_t e = msa::launch_index_merge(cand_score, cand_block, num_shards, T,
                                          cfg->num_groups, cfg->topk, seq_lens, sel, sel_score,
                                          status_word(ws), stream);
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

size_t msa_attn_prefill_workspace(const msa_config_t* cfg, int64_t L) {
  if (check_config(cfg) != MSA_OK || L < 0) return 0;
  if (L == 0) return MSA_WS_HEADER_BYTES;
  return msa::prefill_workspace_layout(L, cfg->num_groups, cfg->topk, prefill_chunk(L)).total;
}

int64_t msa_prefill_chunk_tokens(const msa_config_t* cfg, int64_t L) {
  if (check_config(cfg) != MSA_OK || L <= 0) return 0;
  return prefill_chunk(L);
}

int32_t msa_attn_prefill_launches(const msa_config_t* cfg, int64_t L) {
  if (check_config(cfg) != MSA_OK || L <= 0 || L > kMaxPrefillTokens) return 0;
  const int64_t chunk = prefill_chunk(L);
  return static_cast<int32_t>((L + chunk - 1) / chunk) * msa::prefill_chunk_launches();
}

}  // extern "C"

namespace {

msa_status_t attn_prefill(const msa_config_t* cfg, const void* q, const void* k, const void* v,
                          int64_t L, const int32_t* sel, void* o, float* lse, void* ws,
                          size_t ws_bytes, cudaStream_t stream, cudaEvent_t* marks,
                          int32_t n_marks) {
  msa_status_t st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!q || !k || !v || !sel || !o || !lse || !ws || L < 0) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return MSA_ERR_INVALID_ARG;
  const int G = cfg->num_groups;
  if (cfg->heads_per_group != 16) return MSA_ERR_UNSUPPORTED;
  if (L > kMaxPrefillTokens) return MSA_ERR_UNSUPPORTED;
  if (ws_bytes < msa_attn_prefill_workspace(cfg, L)) return MSA_ERR_WORKSPACE;
  if (L == 0) return MSA_OK;
  const int Hq = G * cfg->heads_per_group;
  CUtensorMap mq, mk, mv;
  {
    const uint64_t dims[3] = {kDim, static_cast<uint64_t>(Hq), static_cast<uint64_t>(L)};
    const uint64_t strides[2] = {kDim * 2, static_cast<uint64_t>(Hq) * kDim * 2};
    const uint32_t box[3] = {64, 16, 1};
    if (!make_map(&mq, q, 3, dims, strides, box)) return MSA_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {kDim, static_cast<uint64_t>(G), static_cast<uint64_t>(L)};
    const uint64_t strides[2] = {kDim * 2, static_cast<uint64_t>(G) * kDim * 2};
    const uint32_t box[3] = {64, 1, kBlock};
    if (!make_map(&mk, k, 3, dims, strides, box)) return MSA_ERR_CUDA;
    if (!make_map(&mv, v, 3, dims, strides, box)) return MSA_ERR_CUDA;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MSA_ERR_CUDA;
  const int64_t chunk = prefill_chunk(L);
  const msa::PrefillWorkspace w = msa::prefill_workspace_layout(L, G, cfg->topk, chunk);
  if (msa::debug_checks_enabled() &&
      msa::debug_check_prefill_sel(sel, L, G, cfg->topk, status_word(ws), stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  int32_t c = 0;
  for (int64_t q0 = 0; q0 < L; q0 += chunk, ++c) {
    MSA_RANGE("prefill_chunk");
    const int64_t q1 = q0 + chunk < L ? q0 + chunk : L;
    cudaEvent_t m3[3] = {nullptr, nullptr, nullptr};
    for (int j = 0; j < 3; ++j)
      if (marks && 3 * c + j < n_marks) m3[j] = marks[3 * c + j];
    cudaError_t e = msa::launch_attn_prefill_chunk(mq, mk, mv, sel, L, G, cfg->topk,
                                                   cfg->softmax_scale, q0, q1,
                                                   static_cast<uint8_t*>(ws), w, o, lse,
                                                   wait_ns(cfg), sms, stream, m3);
    if (e != cudaSuccess) return MSA_ERR_CUDA;
  }
  if (marks && 3 * c < n_marks && marks[3 * c] &&
      cudaEventRecord(marks[3 * c], stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}

}  // namespace

extern "C" {

msa_status_t msa_attn_prefill(const msa_config_t* cfg, const void* q, const void* k,
                              const void* v, int64_t L, const int32_t* sel, void* o, float* lse,
                              void* ws, size_t ws_bytes, cudaStream_t stream) {
  MSA_RANGE("msa_attn_prefill");
  return attn_prefill(cfg, q, k, v, L, sel, o, lse, ws, ws_bytes, stream, nullptr, 0);
}

msa_status_t msa_attn_prefill_marked(const msa_config_t* cfg, const void* q, const void* k,
                                     const void* v, int64_t L, const int32_t* sel, void* o,
                                     float* lse, void* ws, size_t ws_bytes, cudaStream_t stream,
                                     cudaEvent_t* marks, int32_t n_marks) {
  MSA_RANGE("msa_attn_prefill_marked");
  return attn_prefill(cfg, q, k, v, L, sel, o, lse, ws, ws_bytes, stream, marks, n_marks);
}

size_t msa_attn_decode_workspace(const msa_config_t* cfg, const msa_paged_kv_t* paged) {
  if (check_config(cfg) != MSA_OK || !paged || paged->batch < 0) return 0;
  return MSA_WS_HEADER_BYTES +
         align_up(msa::decode_attn_workspace_bytes(paged->batch, cfg->num_groups, cfg->topk),
                  256);
}

msa_status_t msa_attn_decode(const msa_config_t* cfg, const void* q, const msa_paged_kv_t* paged,
                             const int32_t* sel, void* o, float* lse, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
  MSA_RANGE("msa_attn_decode");
  msa_status_t st = check_config(cfg);
  if (st != MSA_OK) return st;
  if ((st = check_paged(paged, true)) != MSA_OK) return st;
  if (!q || !sel || !o || !lse || !ws || !aligned16(q) || !aligned16(o)) return MSA_ERR_INVALID_ARG;
  if (cfg->heads_per_group != 16) return MSA_ERR_UNSUPPORTED;
  if (ws_bytes < msa_attn_decode_workspace(cfg, paged)) return MSA_ERR_WORKSPACE;
  if (paged->batch == 0) return MSA_OK;
  const int G = cfg->num_groups;
  const bool kv8 = paged->kv_dtype == MSA_KV_E4M3;
  CUtensorMap mk, mv;
  {
    // rows of 128 elements: two 64-element bf16 panels, or one 128-byte e4m3 box
    const uint64_t dims[2] = {kDim, static_cast<uint64_t>(paged->num_pages) * G * kBlock};
    const uint64_t strides[1] = {kDim * (kv8 ? 1u : 2u)};
    const uint32_t box[2] = {kv8 ? 128u : 64u, kBlock};
    const CUtensorMapDataType t =
        kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!msa::encode_tmap(&mk, t, paged->k_pool, 2, dims, strides, box) ||
        !msa::encode_tmap(&mv, t, paged->v_pool, 2, dims, strides, box))
      return MSA_ERR_CUDA;
  }
  int sms = 0;
  if (!sm_count(&sms)) return MSA_ERR_CUDA;
  if (msa::debug_checks_enabled() &&
      (msa::debug_check_paged(paged->page_table, paged->seq_lens, paged->batch, paged->max_pages,
                              paged->num_pages, status_word(ws), stream) != cudaSuccess ||
       msa::debug_check_decode_sel(sel, paged->seq_lens, paged->batch, G, cfg->topk,
                                   paged->max_pages, status_word(ws), stream) != cudaSuccess))
    return MSA_ERR_CUDA;
  cudaError_t e = msa::launch_decode_attn(
      mk, mv, q, sel, paged->page_table, paged->seq_lens, paged->batch, paged->max_pages,
      paged->num_pages, G, cfg->topk, cfg->softmax_scale,
      static_cast<uint8_t*>(ws) + MSA_WS_HEADER_BYTES, o, lse, status_word(ws), wait_ns(cfg), sms,
      stream, kv8);
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // extern "C"
