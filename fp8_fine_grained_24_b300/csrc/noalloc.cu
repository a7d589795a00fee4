// fp8_gemm_dense_noalloc: the dense FP8 GEMM for callers that cannot
// allocate device memory.
//
// fp8_gemm_dense asks its caller for a scratch buffer when it splits K for
// decode-sized problems. Some callers have no way to provide one: a plug-in
// or operator library that is handed device pointers by a host application
// which owns every byte of device memory and exposes no allocator; code on a
// latency-critical loop where a device allocation (which can synchronize the
// whole device) is forbidden; an embedded deployment that must know, when the
// library is loaded, exactly how much device memory it will ever hold.
//
// This entry point takes the same inputs and outputs as fp8_gemm_dense and
// no workspace. Its scratch is a fixed array in device memory that the
// library reserves when it is loaded: 64 MiB on every GPU the process uses,
// held until the process exits. That covers every dense shape on GPUs with
// up to about 170 SMs (the Stream-K scratch holds at most three 128 KB
// partial tiles per SM plus counters). Nothing here calls
// cudaMalloc, cudaFree or any routine that allocates.
//
// Notes for users:
//   * The first call on a device does the set-up: it looks up the array's
//     device address on that device (cudaGetSymbolAddress) and caches it.
//     That first call should come before any stream capture.
//   * All calls in the process share the one array. Two calls whose GPU work
//     overlaps (different streams, or different host threads without
//     ordering) race on it and may produce wrong results: order them.
//   * A problem whose scratch need exceeds the array is rejected with
//     FP8FG_ERR_UNSUPPORTED_SHAPE before anything is enqueued.
//   * The part of the scratch that must start at zero (the Stream-K arrival
//     counters) is cleared on the caller's stream by every call.
#include <mutex>

#include "../../include/fp8fg.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = 64u << 20;  // 64 MiB per device

// The scratch itself. In host code this name is only a host-side stand-in:
// its device address comes from cudaGetSymbolAddress (below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kStaticScratchBytes];

struct NoallocDevice {
  bool ready = false;
  void* scratch = nullptr;
  int num_sms = 0;
};
NoallocDevice g_noalloc[64];
std::mutex g_noalloc_mu;

// Set-up once per device, with that device current.
int noalloc_device(NoallocDevice** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    fp8fg::set_last_error("fp8_gemm_dense_noalloc: cudaGetDevice failed");
    return FP8FG_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocDevice& d = g_noalloc[dev];
  if (!d.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      fp8fg::set_last_error("fp8_gemm_dense_noalloc: cudaGetSymbolAddress(static scratch) failed");
      return FP8FG_ERR_CUDA;
    }
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      fp8fg::set_last_error("fp8_gemm_dense_noalloc: cudaDeviceGetAttribute failed");
      return FP8FG_ERR_CUDA;
    }
    d.scratch = p;
    d.ready = true;
  }
  *out = &d;
  return FP8FG_OK;
}

}  // namespace

extern "C" {

int fp8_gemm_dense_noalloc(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                           int b_scale_kind, void* C, int out_dtype, int accumulate, int64_t M, int64_t N,
                           int64_t K, fp8fg_stream_t stream) {
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool plausible = M > 0 && N > 0 && K > 0 && K % 128 == 0 && N % 8 == 0 && M < (1ll << 31) &&
                         N < (1ll << 31) && K < (1ll << 31) && A && sA && B && sB && C && a16(A) && a16(B) &&
                         a16(C) && a16(sA) && (b_scale_kind == FP8FG_SCALE_BLOCK128 || b_scale_kind == FP8FG_SCALE_ROW) &&
                         (out_dtype == FP8FG_BF16 || out_dtype == FP8FG_FP32) && (accumulate == 0 || accumulate == 1) &&
                         !(accumulate && out_dtype != FP8FG_FP32) &&
                         (reinterpret_cast<uintptr_t>(sB) & (b_scale_kind == FP8FG_SCALE_ROW ? 15u : 3u)) == 0;
  if (!plausible) {
    // empty or rejected arguments: the dense entry point gives the answer (a
    // no-op or its error code and message) and nothing is enqueued here
    return fp8_gemm_dense(A, sA, B, sB, b_scale_kind, C, out_dtype, accumulate, M, N, K, nullptr, 0, stream);
  }
  NoallocDevice* d = nullptr;
  int rc = noalloc_device(&d);
  if (rc != FP8FG_OK) return rc;
  const size_t need = fp8fg::gemm_workspace_bytes(fp8fg::kModeDense, M, N, K, 1, d->num_sms);
  if (need > kStaticScratchBytes) {
    fp8fg::set_last_error(
        "fp8_gemm_dense_noalloc: this shape needs more Stream-K scratch than the library's static 64 MiB "
        "array; use fp8_gemm_dense with a workspace");
    return FP8FG_ERR_UNSUPPORTED_SHAPE;
  }
  if (need > 0) {
    size_t off = 0, bytes = 0;
    fp8fg::gemm_workspace_zero_range(fp8fg::kModeDense, M, N, K, 1, d->num_sms, kStaticScratchBytes, &off, &bytes);
    if (bytes > 0) {
      cudaError_t e = cudaMemsetAsync(static_cast<unsigned char*>(d->scratch) + off, 0, bytes,
                                      reinterpret_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) {
        fp8fg::set_last_error("fp8_gemm_dense_noalloc: clearing the scratch counters failed");
        return FP8FG_ERR_CUDA;
      }
    }
  }
  return fp8_gemm_dense(A, sA, B, sB, b_scale_kind, C, out_dtype, accumulate, M, N, K, d->scratch,
                        kStaticScratchBytes, stream);
}

}  // extern "C"
