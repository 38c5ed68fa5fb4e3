// Tensor-map (TMA descriptor) encoding shared by the host side of the MSA kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace msa {

// Tiled tensor map, with the 128-byte swizzle unless swizzle128 is false (then the box lands in
// shared memory densely, innermost dimension first).  dims / box innermost first; strides in bytes
// for dimensions 1..rank-1.  Returns false if the driver entry point is missing or rejects the map.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                 const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                 bool swizzle128 = true);

}  // namespace msa
