/*
 * msa.h — C ABI of libmsa, the MiniMax Sparse Attention (MSA) operator for GB300 (sm_103a).
 *
 * MSA is defined on the page "MiniMax M3 算力省 20 倍" (mizuki-eaf.pages.dev), section 二:
 *   - Index Branch: each GQA group has one index-query head, all groups share one index-key head.
 *     Index scores are raw query·key dot products over the causal window, max-pooled into
 *     B-token block scores; every group picks its own top-k blocks; the query's own (local)
 *     block is always picked (section 三 item 4: it keeps a reserved slot, so it counts in k).
 *   - Main Branch: exact softmax attention over the tokens of the selected blocks only,
 *     causal inside the local block.  Deployment: B = 128, k = 16 (2048 keys per query).
 * Decode over a paged KV cache is named on the page "MiniMax M3 的采用瓶颈，会卡在 serving 生态"
 * (paragraph on Together AI: paged MSA decode, KV-block-major sparse attention).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers, owned by the caller; the library never allocates
 *     and never frees.  Tensors are dense, row-major, in the layouts stated per argument.
 *   - bf16 means IEEE bfloat16 bits (uint16).  Pointers passed to TMA-fed kernels must be
 *     16-byte aligned (q, k, v, q_idx, k_idx and the pools); violations return INVALID_ARG.
 *   - Every call is asynchronous on `stream` and never synchronizes, except
 *     msa_get_device_status.  Calls are stateless and thread-safe; concurrent calls must not
 *     share a workspace.
 *   - `ws` is caller-owned device scratch of at least the size the matching *_workspace()
 *     query returns (never less than MSA_WS_HEADER_BYTES).  Its first MSA_WS_HEADER_BYTES hold a
 *     device status word: zero it once before first use (msa_reset_device_status or a memset);
 *     kernels record the first device-side error there (a bounded wait that ran out, an index
 *     out of range) and it stays set until reset.  Device-side errors never trap: the kernel
 *     skips the offending access and finishes.
 *   - Host-side argument errors return before anything is enqueued.  Launch failures return
 *     MSA_ERR_CUDA.
 *   - Tracing: a library built with MSA_NVTX (the default build) wraps every call that enqueues
 *     work in an NVTX range named after the call (and each 64K-query pass of the prefill main
 *     branch in a nested range "prefill_chunk"), so profilers can select one call's kernels.
 *   - Checked build: libmsa_debug.so, compiled with MSA_DEBUG_CHECKS, exports the same calls.
 *     Its kernels check the indices they derive (schedule positions, work items, listed tokens,
 *     scanned pages, written rows) before each access, clamp or skip a failing one, flag
 *     MSA_ERR_DEVICE_BOUNDS and record the first failure (msa_get_debug_record).  With the
 *     environment variable MSA_DEBUG_CHECKS set (to anything but "" or "0") it also validates
 *     the caller's index tensors before the kernels run: selection rows in the form
 *     msa_index_select writes them (ascending, within the query's causal range, the query's own
 *     block present, -1 only as trailing padding), sequence lengths in [1, max_pages * 128] and
 *     every page-table entry of a used page in [0, num_pages).  Results are bit-identical to the
 *     release build's when no check fails.
 *   - v1 supports head_dim = index_dim = block_size = 128, 1 <= topk <= 16, num_groups <= 4 for
 *     the index branch (any number of groups for the main branch), heads_per_group = 16 for the
 *     main branch (prefill and decode: a group's 16 query heads are the rows of its tensor-core
 *     tiles), prefill lengths up to 1,572,864; other values return MSA_ERR_UNSUPPORTED.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Workspace header: bytes [0, 4) the device status word; bytes [16, 48) the checked build's
 * msa_debug_record_t; the rest is reserved. */
#define MSA_WS_HEADER_BYTES 256

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size, inconsistent config */
  MSA_ERR_UNSUPPORTED = 2,    /* a size this build does not implement */
  MSA_ERR_WORKSPACE = 3,      /* ws_bytes smaller than the *_workspace() query */
  MSA_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
  MSA_ERR_DEVICE_TIMEOUT = 5, /* device status: a bounded wait ran out */
  MSA_ERR_DEVICE_BOUNDS = 6   /* device status: a page id or block id was out of range */
} msa_status_t;

/* Element type of the index vectors (q_idx, k_idx, the paged k_idx_pool).  E4M3 is the OCP
 * 8-bit float (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities): the
 * indexer's QK product in FP8, as the pages' Blackwell kernel computes it ("MiniMax M3.1 Flash
 * 开放权重与部署要点", section 权重能下载之后，为什么还要先看 vLLM, where FP8 is the compute type
 * NVFP4-stored keys are dequantised to).  Scores accumulate in fp32 either way; e4m3 halves the
 * index bytes and doubles the tensor-core rate. */
typedef enum { MSA_INDEX_BF16 = 0, MSA_INDEX_E4M3 = 1 } msa_index_dtype_t;

/* Element type of the paged K and V pools.  E4M3 is the same OCP 8-bit float: an FP8 KV cache
 * ("MiniMax M3.1 Flash 开放权重与部署要点", section 稀疏注意力为什么还会撞上显存墙, where the
 * FP8 cache halves the bytes per token), read by the decode attention and widened exactly in
 * the kernel (to bf16 for q.K, to fp16 for P.V).  The values are used as stored: no scale. */
typedef enum { MSA_KV_BF16 = 0, MSA_KV_E4M3 = 1 } msa_kv_dtype_t;

typedef struct {
  int32_t num_groups;      /* G: KV heads = GQA groups = index-query heads */
  int32_t heads_per_group; /* query heads per group; Hq = G * heads_per_group */
  int32_t head_dim;        /* d of q/k/v (128) */
  int32_t index_dim;       /* d_i of the index query/key heads (128) */
  int32_t block_size;      /* B (128) */
  int32_t topk;            /* k, the local block included (1..16) */
  float softmax_scale;     /* multiplies q.k in the main branch (1/sqrt(d) in the tests) */
  int32_t index_dtype;     /* msa_index_dtype_t of q_idx, k_idx and k_idx_pool (0: bf16) */
  int64_t wait_limit_ns;   /* bound on every device-side wait; 0 selects 2 seconds */
} msa_config_t;

/* A paged KV cache of B-token pages shared by `batch` sequences.  Logical block b of sequence s
 * lives in physical page page_table[s*max_pages + b]. */
typedef struct {
  const void* k_idx_pool;    /* index_dtype [num_pages][B][d_i]: index keys */
  const void* k_pool;        /* kv_dtype [num_pages][G][B][d]: keys, head-major inside a page */
  const void* v_pool;        /* kv_dtype [num_pages][G][B][d]: values, same layout */
  const int32_t* page_table; /* int32 [batch][max_pages], device */
  const int32_t* seq_lens;   /* int32 [batch], device: context length n >= 1 per sequence; the
                                query is the token at n-1, already written to the cache */
  int32_t batch;
  int32_t max_pages;         /* row length of page_table; n <= max_pages * B is required */
  int32_t num_pages;         /* pool size; page ids must lie in [0, num_pages) */
  int32_t kv_dtype;          /* msa_kv_dtype_t of k_pool and v_pool (0: bf16) */
} msa_paged_kv_t;

/* Workspace bytes for msa_index_select: num_queries = L for prefill (paged == NULL), the batch
 * for decode (paged != NULL, num_keys ignored). */
size_t msa_index_select_workspace(const msa_config_t* cfg, int64_t num_queries, int64_t num_keys,
                                  const msa_paged_kv_t* paged);

/*
 * Index branch: block scores, max-pooling, per-group top-k with the forced local block.
 *   Prefill (paged == NULL): q_idx [L][G][d_i] (query i is the token at position i),
 *     k_idx [L][d_i].  Output rows: T = L.
 *   Decode (paged != NULL, k_idx and L ignored): q_idx [batch][G][d_i], one query per
 *     sequence at position seq_lens[s]-1; index keys read from paged->k_idx_pool.  T = batch.
 *   Index vectors are bf16 or e4m3 as cfg->index_dtype says.
 *   sel (out) int32 [G][T][k]: selected block ids, ascending, padded with -1 when fewer than k
 *     blocks exist.  Ranking is by raw score (higher first), ties to the lower block id.
 *   sel_score (out, optional, may be NULL) fp32 [G][T][k]: the pooled score of each selected
 *     block; +inf for the local block (it is never scored), -inf for padding.
 */
msa_status_t msa_index_select(const msa_config_t* cfg, const void* q_idx, const void* k_idx,
                              int64_t L, const msa_paged_kv_t* paged, int32_t* sel,
                              float* sel_score, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Index branch with every block's pooled score exported, for the KL alignment of the indexer
 * ("MiniMax M3 算力省 20 倍", section 三 item 1: the indexer's block distribution is fitted to the
 * main branch's group-mean attention; that loss and its gradient live outside this library).
 * Same arguments, workspace and outputs as msa_index_select, plus
 *   block_scores (out, required) fp32, prefill [G][L][nb] with nb = ceil(L / B), decode
 *     [G][batch][max_pages]: for query i in block b(i) and every block c < b(i) the max-pooled
 *     raw score max over j in c of q_idx[i,g] . k_idx[j]; +inf at c = b(i) (the forced local
 *     block, never scored); -inf for c > b(i) (not causal).  A decode row whose seq_lens entry
 *     is out of range (MSA_ERR_DEVICE_BOUNDS) is all -inf.  The scores are bit-identical to the
 *     ones that msa_index_select ranks.
 * Returns MSA_ERR_INVALID_ARG if block_scores is NULL.
 */
msa_status_t msa_index_select_scores(const msa_config_t* cfg, const void* q_idx,
                                     const void* k_idx, int64_t L, const msa_paged_kv_t* paged,
                                     int32_t* sel, float* sel_score, float* block_scores,
                                     void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Context-parallel index branch, step 1 of 2: the candidates of one shard of the key blocks.
 * The pages describe the indexer's decode running context-parallel over several GPUs
 * ("MiniMax M3.1 Flash 开放权重与部署要点", section 权重能下载之后，为什么还要先看 vLLM: 4 GB300 at
 * 512K context).  Each GPU holds the index keys of a range of blocks, ranks its own blocks and
 * keeps its top-(k-1); the candidates of all shards are exchanged (an all-gather of
 * (k-1) x (4 + 4) bytes per (query, group)) and msa_index_merge ranks them into the selection.
 * Every block of the global top-(k-1) is within its own shard's top-(k-1), so the merged
 * selection equals msa_index_select's bit for bit when the shards cover [0, nb) without overlap.
 *   Shard: logical key blocks [block_begin, block_end) (clamped to the sequence); only blocks
 *     strictly before a query's own block are ranked for it (the local block is added by the
 *     merge).
 *   Prefill (paged == NULL): q_idx [L][G][d_i] (all queries); k_idx holds the index keys of the
 *     shard only, positions [block_begin*B, min(block_end*B, L)) as [rows][d_i]; L is the whole
 *     sequence length.  T = L.
 *   Decode (paged != NULL, k_idx and L ignored): q_idx [batch][G][d_i]; only the page-table
 *     entries of blocks in the shard are read.  T = batch.
 *   cand_score (out) fp32 [G][T][k-1], cand_block (out) int32 [G][T][k-1]: the shard's
 *     top-(k-1) in rank order (score desc, block asc), padded with (-inf, -1).  With k = 1 there
 *     is nothing to write and both may be NULL.
 *   ws / ws_bytes: as for msa_index_select with the same arguments.
 */
msa_status_t msa_index_candidates(const msa_config_t* cfg, const void* q_idx, const void* k_idx,
                                  int64_t L, const msa_paged_kv_t* paged, int32_t block_begin,
                                  int32_t block_end, float* cand_score, int32_t* cand_block,
                                  void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Context-parallel index branch, step 2 of 2: the selection from the candidates of num_shards
 * disjoint shards, stacked as cand_score / cand_block [num_shards][G][T][k-1] (the all-gather's
 * output).  Ranks the union by (score desc, block asc), keeps min(k-1, blocks before the
 * query's own) of them, adds the local block and writes sel [G][T][k] ascending, -1 padded
 * (sel_score optional, as msa_index_select writes it).
 *   seq_lens (device, int32 [T]): decode, query t is the token at seq_lens[t]-1; NULL: prefill,
 *     query t is the token at position t.
 *   ws: at least MSA_WS_HEADER_BYTES; a candidate at or after its query's own block, or a
 *     context length <= 0, is skipped and flagged as MSA_ERR_DEVICE_BOUNDS.
 */
msa_status_t msa_index_merge(const msa_config_t* cfg, int32_t num_shards,
                             const float* cand_score, const int32_t* cand_block, int64_t T,
                             const int32_t* seq_lens, int32_t* sel, float* sel_score, void* ws,
                             size_t ws_bytes, cudaStream_t stream);

/* Workspace bytes for msa_attn_prefill over L tokens. */
size_t msa_attn_prefill_workspace(const msa_config_t* cfg, int64_t L);

/*
 * Main branch, prefill: exact softmax attention of every query head over the tokens of its
 * group's selected blocks, causal inside the local block (KV-outer order with a two-phase
 * log-sum-exp combine; results do not depend on scheduling).
 *   q bf16 [L][Hq][d]; k, v bf16 [L][G][d]; sel int32 [G][L][k] as msa_index_select writes it.
 *   o (out) bf16 [L][Hq][d]; lse (out) fp32 [Hq][L], natural log of the softmax denominator of
 *   the scaled logits.  Ids in sel outside [0, block of the query] are skipped and flagged as
 *   MSA_ERR_DEVICE_BOUNDS in the status word.
 */
msa_status_t msa_attn_prefill(const msa_config_t* cfg, const void* q, const void* k,
                              const void* v, int64_t L, const int32_t* sel, void* o, float* lse,
                              void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Instrumented form of msa_attn_prefill, for timing its phases; results are identical.
 * marks (may be NULL) are caller-created CUDA events (timing enabled).  On `stream` the call
 * records, for query chunk c: marks[3c] before the scheduling kernels, marks[3c+1] before the
 * attention kernel, marks[3c+2] before the combine kernel, and marks[3*chunks] after the last
 * combine.  Recording stops after n_marks events.  Chunks are msa_prefill_chunk_tokens() long.
 */
msa_status_t msa_attn_prefill_marked(const msa_config_t* cfg, const void* q, const void* k,
                                     const void* v, int64_t L, const int32_t* sel, void* o,
                                     float* lse, void* ws, size_t ws_bytes, cudaStream_t stream,
                                     cudaEvent_t* marks, int32_t n_marks);

/* Query tokens per main-branch pass of msa_attn_prefill (its workspace covers one pass). */
int64_t msa_prefill_chunk_tokens(const msa_config_t* cfg, int64_t L);

/* Kernel launches one msa_attn_prefill call of length L enqueues (for launch accounting; 0 for
 * invalid arguments).  No GPU work. */
int32_t msa_attn_prefill_launches(const msa_config_t* cfg, int64_t L);

/*
 * msa_attn_prefill_noalloc — msa_attn_prefill for callers that cannot allocate device memory.
 * (The method's description has no counterpart: this is a deployment convenience of this
 * library.)
 *
 * Some callers are handed only their input and output tensors and are not allowed to allocate:
 * a plugin or callback inside another framework's memory pool, code on a latency-critical path
 * where cudaMalloc (which can synchronize the device) is forbidden, or an engine whose device
 * memory budget is fixed ahead of time.  This entry point needs no workspace from them: its
 * scratch is a library-owned static device array of MSA_NOALLOC_SCRATCH_BYTES (64 MiB), which
 * every GPU that loads libmsa holds until the process exits.  The call itself allocates nothing
 * (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 *   Arguments are those of msa_attn_prefill without ws/ws_bytes; outputs are identical.
 *   device_status (optional, device pointer to one int32): receives the device status word of
 *     this call (0, MSA_ERR_DEVICE_TIMEOUT or MSA_ERR_DEVICE_BOUNDS) when the call's work has run.
 *   Queries are processed in passes sized to fit the scratch (128 queries per pass at G = 4,
 *     k = 16), so long prefills run slower than msa_attn_prefill with a full workspace.
 *   Sizes beyond what the scratch or the kernels can take (L above 1,572,864 tokens, or a
 *     configuration whose 128-query pass would not fit) return MSA_ERR_UNSUPPORTED before
 *     anything is enqueued.
 *   The first call on each device looks up the device address of the scratch array
 *     (cudaGetSymbolAddress, with that device current); make that first call before any stream
 *     capture.
 *   All calls share the one array, which keeps the last call's contents; the call clears what
 *     must start at zero.  Calls that overlap on the GPU (different streams, concurrent host
 *     threads) race on it: issue them in order on one stream.
 */
#define MSA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
msa_status_t msa_attn_prefill_noalloc(const msa_config_t* cfg, const void* q, const void* k,
                                      const void* v, int64_t L, const int32_t* sel, void* o,
                                      float* lse, int32_t* device_status, cudaStream_t stream);

/* Workspace bytes for msa_attn_decode on this cache shape. */
size_t msa_attn_decode_workspace(const msa_config_t* cfg, const msa_paged_kv_t* paged);

/*
 * Main branch, paged decode: one query token per sequence at position seq_lens[s]-1.
 *   q bf16 [batch][Hq][d]; sel int32 [G][batch][k] (logical block ids, as msa_index_select
 *   writes them).  o (out) bf16 [batch][Hq][d]; lse (out) fp32 [Hq][batch].
 *   Page ids outside [0, num_pages) and block ids outside [0, block of the query] are skipped
 *   and flagged as MSA_ERR_DEVICE_BOUNDS.
 */
msa_status_t msa_attn_decode(const msa_config_t* cfg, const void* q,
                             const msa_paged_kv_t* paged, const int32_t* sel, void* o,
                             float* lse, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronizes `stream`, then returns the device status recorded in ws (MSA_OK if none). */
msa_status_t msa_get_device_status(const void* ws, cudaStream_t stream);

/* Enqueues a clear of the device status word in ws, and of the checked build's record, on
 * `stream`. */
msa_status_t msa_reset_device_status(void* ws, cudaStream_t stream);

/* The checks of the checked build (libmsa_debug.so), each named by the site that failed. */
typedef enum {
  MSA_SITE_NONE = 0,
  /* the caller's index tensors (validated when MSA_DEBUG_CHECKS is set in the environment) */
  MSA_SITE_SEL_RANGE = 1,    /* a selected id outside [-1, block of the query]:
                                value = the id, bound = that block + 1 */
  MSA_SITE_SEL_ORDER = 2,    /* ids not strictly ascending, or an id after -1 padding:
                                value = the slot, bound = k */
  MSA_SITE_SEL_LOCAL = 3,    /* the query's own block missing: value = the row's last id */
  MSA_SITE_SEQ_LEN = 4,      /* seq_lens[s] outside [1, max_pages * 128]: row = s */
  MSA_SITE_PAGE_ID = 5,      /* a used page's page-table entry outside [0, num_pages): row = s */
  /* indices the kernels derive, checked before each access */
  MSA_SITE_SCHED_LIST = 16,  /* a (token, slot) list position past the pass's units */
  MSA_SITE_SCHED_ITEM = 17,  /* a work item past the workspace's item capacity */
  MSA_SITE_ATTN_ITEM = 18,   /* a work item's group, block, token count or list range */
  MSA_SITE_ATTN_TOKEN = 19,  /* a listed token outside the pass or before the item's block */
  MSA_SITE_COMBINE_POS = 20, /* a slot's list position past the pass's units */
  MSA_SITE_DECODE_PAGE = 21, /* a scanned (sequence, logical page) outside the batch's range */
  MSA_SITE_INDEX_ROW = 22    /* a selection row's group, or a kept block the row did not score */
} msa_debug_site_t;

/* The first failed check since the last reset.  row names what the failure concerns: g * T + t
 * for a selection row of query t in group g (T = L or batch), the sequence for paged input, the
 * query or work item for the kernels' own checks. */
typedef struct {
  int32_t site;     /* msa_debug_site_t; MSA_SITE_NONE if no check failed */
  int32_t reserved;
  int64_t value;    /* the offending value */
  int64_t bound;    /* the exclusive upper bound of the check */
  int64_t row;
} msa_debug_record_t;

/* 0 for the release build; in the checked build bit 0 is set, and bit 1 when the caller's index
 * tensors are validated (MSA_DEBUG_CHECKS set in the environment). */
int32_t msa_debug_checks(void);

/* Synchronizes `stream`, then copies the record of the first failed check from ws.  The release
 * build keeps no record: it zeroes *record and returns MSA_ERR_UNSUPPORTED. */
msa_status_t msa_get_debug_record(const void* ws, msa_debug_record_t* record,
                                  cudaStream_t stream);

/* Static description of a status code. */
const char* msa_status_string(msa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
