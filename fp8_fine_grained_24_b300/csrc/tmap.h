// Host-side TMA tensor-map encoding shared by the GEMM and the quantizers.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fp8fg {

// Encode a tiled tensor map of rank 3: dims {d0, d1, d2} (d0 contiguous),
// byte strides {stride1, stride2} of dims 1 and 2, box {b0, b1, 1}, element
// strides 1, out-of-bounds elements read as zero. False when the driver
// entry point is missing or the driver rejects the arguments.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw);

// Rank 4: dims (dims[0] contiguous), byte strides of dims 1..3, box. A box
// lands in shared memory densely in dimension order when sw is
// CU_TENSOR_MAP_SWIZZLE_NONE; with a swizzle, every innermost row takes a
// whole swizzle span even when it is shorter.
bool make_map4(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[4],
               const uint64_t (&strides)[3], const uint32_t (&box)[4], CUtensorMapSwizzle sw);

}  // namespace fp8fg
