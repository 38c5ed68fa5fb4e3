// NVTX ranges around the C-ABI calls (compiled in with MSA_NVTX): each call is one named range
// on the calling thread, so a profiler can filter the kernels of one call (for instance
// `ncu --nvtx --nvtx-include "msa_attn_prefill/"`).  NVTX v3 is header-only; without an attached
// tool a range costs a branch on a null function pointer.
#pragma once

#if defined(MSA_NVTX)
#include <nvtx3/nvToolsExt.h>

namespace msa {
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace msa

#define MSA_RANGE_CAT2(a, b) a##b
#define MSA_RANGE_CAT(a, b) MSA_RANGE_CAT2(a, b)
#define MSA_RANGE(name) ::msa::NvtxRange MSA_RANGE_CAT(msa_nvtx_range_, __LINE__)(name)
#else
#define MSA_RANGE(name) static_cast<void>(0)
#endif
