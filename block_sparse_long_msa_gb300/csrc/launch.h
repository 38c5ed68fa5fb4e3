// Internal launch entry points of the MSA kernels (host side, C++).  The public C ABI in
// include/msa.h validates arguments and builds tensor maps, then calls these.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace msa {

size_t index_prefill_smem_bytes(int G, int ns);
cudaError_t launch_index_select_prefill(const CUtensorMap& map_q, const CUtensorMap& map_k,
                                        int64_t L, int G, int k, int32_t* sel, float* sel_score,
                                        int32_t* status, uint64_t wait_ns, cudaStream_t stream);

}  // namespace msa
