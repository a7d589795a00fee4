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

}  // namespace fp8fg
