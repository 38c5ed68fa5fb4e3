// msa_attn_prefill_noalloc: the prefill main branch for callers that cannot allocate device
// memory.  Its scratch is a library-owned static device array instead of a caller workspace;
// the kernels and their arithmetic are those of msa_attn_prefill.
#include <mutex>

#include "../../include/msa.h"
#include "common.cuh"
#include "launch.h"
#include "tmap.h"
#include "trace.h"

namespace {

constexpr size_t kScratchBytes = MSA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxTokens = 1536 * 1024;  // same limit as msa_attn_prefill

}  // namespace

// One copy per GPU that loads this library, held until the process exits.  In host code the
// name is only a stand-in: the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

namespace {

struct DeviceScratch {
  std::mutex mu;
  void* ptr = nullptr;  // set once the lookup has succeeded on this device
};
DeviceScratch g_scratch[kMaxDevices];

// Set-up, once per device, with that device current: the device address of the scratch array.
// Only a successful lookup is kept; a failed one (for example made while the stream was being
// captured) clears the runtime's last error and is tried again by the next call.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceScratch& s = g_scratch[dev];
  std::lock_guard<std::mutex> lock(s.mu);
  if (!s.ptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) == cudaSuccess) {
      s.ptr = p;
    } else {
      (void)cudaGetLastError();
    }
  }
  return s.ptr;
}

bool encode_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint32_t b1, uint32_t b2) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const uint32_t box[3] = {64, b1, b2};
  return msa::encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, 3, dims, strides, box);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" msa_status_t msa_attn_prefill_noalloc(const msa_config_t* cfg, const void* q,
                                                 const void* k, const void* v, int64_t L,
                                                 const int32_t* sel, void* o, float* lse,
                                                 int32_t* device_status, cudaStream_t stream) {
  MSA_RANGE("msa_attn_prefill_noalloc");
  if (!cfg || cfg->num_groups < 1 || cfg->heads_per_group < 1 || cfg->topk < 1 ||
      (cfg->index_dtype != MSA_INDEX_BF16 && cfg->index_dtype != MSA_INDEX_E4M3) ||
      cfg->wait_limit_ns < 0 || !(cfg->softmax_scale == cfg->softmax_scale))
    return MSA_ERR_INVALID_ARG;
  if (cfg->head_dim != msa::kDim || cfg->index_dim != msa::kDim ||
      cfg->block_size != msa::kBlock || cfg->topk > msa::kTopMax || cfg->heads_per_group != 16)
    return MSA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !sel || !o || !lse || L < 0) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return MSA_ERR_INVALID_ARG;
  if (L > kMaxTokens) return MSA_ERR_UNSUPPORTED;
  const int G = cfg->num_groups, topk = cfg->topk;
  // largest multiple of 128 queries per pass whose scratch fits the static array
  int64_t chunk = (L + msa::kBlock - 1) / msa::kBlock * msa::kBlock;
  if (chunk > 65536) chunk = 65536;
  while (chunk >= msa::kBlock &&
         msa::prefill_workspace_layout(L > 0 ? L : 1, G, topk, chunk).total > kScratchBytes)
    chunk -= msa::kBlock;
  if (chunk < msa::kBlock) return MSA_ERR_UNSUPPORTED;  // one 128-query pass does not fit
  if (L == 0) return MSA_OK;

  uint8_t* scratch = static_cast<uint8_t*>(scratch_on_current_device());
  if (!scratch) return MSA_ERR_CUDA;
  const int Hq = G * cfg->heads_per_group;
  CUtensorMap mq, mk, mv;
  if (!encode_3d(&mq, q, msa::kDim, Hq, L, 16, 1) ||
      !encode_3d(&mk, k, msa::kDim, G, L, 1, msa::kBlock) ||
      !encode_3d(&mv, v, msa::kDim, G, L, 1, msa::kBlock))
    return MSA_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MSA_ERR_CUDA;
  // the status word in the scratch header starts every call at zero; the rest of the scratch is
  // fully written by the scheduling kernels before it is read
  if (cudaMemsetAsync(scratch, 0, MSA_WS_HEADER_BYTES, stream) != cudaSuccess) return MSA_ERR_CUDA;
  const uint64_t wait_ns = cfg->wait_limit_ns > 0 ? static_cast<uint64_t>(cfg->wait_limit_ns)
                                                  : msa::kDefaultWaitNs;
  const msa::PrefillWorkspace w = msa::prefill_workspace_layout(L, G, topk, chunk);
  if (msa::debug_checks_enabled() &&
      msa::debug_check_prefill_sel(sel, L, G, topk, reinterpret_cast<int32_t*>(scratch),
                                   stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  for (int64_t q0 = 0; q0 < L; q0 += chunk) {
    const int64_t q1 = q0 + chunk < L ? q0 + chunk : L;
    cudaEvent_t none[3] = {nullptr, nullptr, nullptr};
    if (msa::launch_attn_prefill_chunk(mq, mk, mv, sel, L, G, topk, cfg->softmax_scale, q0, q1,
                                       scratch, w, o, lse, wait_ns, sms, stream,
                                       none) != cudaSuccess)
      return MSA_ERR_CUDA;
  }
  if (device_status && cudaMemcpyAsync(device_status, scratch, sizeof(int32_t),
                                       cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}
