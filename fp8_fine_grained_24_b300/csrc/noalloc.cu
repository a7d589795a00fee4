// fp8_gemm_dense_noalloc: the dense FP8 GEMM for callers that cannot
// allocate device memory.
//
// fp8_gemm_dense asks its caller for a scratch buffer for decode-sized
// problems, which its Stream-K split sums partial tiles in (its cluster
// split, the default where it applies, needs none). Some callers have no
// way to provide one: a plug-in
// or operator library that is handed device pointers by a host application
// which owns every byte of device memory and exposes no allocator; code on a
// latency-critical loop where a device allocation (which can synchronize the
// whole device) is forbidden; an embedded deployment that must know, when the
// library is loaded, exactly how much device memory it will ever hold.
//
// This entry point takes the same inputs and outputs as fp8_gemm_dense and
// no workspace. Its scratch is a fixed 64 MiB array in device memory, part
// of this library's device code. That covers every dense shape on GPUs with
// up to about 170 SMs (the Stream-K scratch holds at most three 128 KB
// partial tiles per SM plus counters). Nothing here calls cudaMalloc,
// cudaFree or any routine that allocates.
//
// Notes for users:
//   * When the memory is committed: the CUDA runtime loads a library's
//     device code lazily by default (CUDA_MODULE_LOADING=LAZY), so the
//     array is committed on a device by the first call of this entry point
//     there, which looks up its device address (cudaGetSymbolAddress) and
//     caches it. That first call may therefore fail for lack of device
//     memory, and it may synchronize the device: make it once at start-up,
//     outside any latency-critical region and before any stream capture.
//     From then on the array stays held on that device until the process
//     exits. (With CUDA_MODULE_LOADING=EAGER it is committed when the
//     library is loaded.)
//   * All calls in the process share the one array. Two calls whose GPU work
//     overlaps (different streams, or different host threads without
//     ordering) race on it and may produce wrong results: order them.
//   * Arguments are checked exactly as fp8_gemm_dense checks them, on the
//     host, before anything is enqueued. A problem whose scratch need
//     exceeds the array is rejected with FP8FG_ERR_UNSUPPORTED_SHAPE.
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
  if (M == 0 || N == 0) {
    // empty product: the dense entry point's answer (a no-op, or its error
    // for negative sizes); nothing is enqueued
    return fp8_gemm_dense(A, sA, B, sB, b_scale_kind, C, out_dtype, accumulate, M, N, K, nullptr, 0, stream);
  }
  int rc = fp8fg::check_gemm_common(A, sA, B, sB, b_scale_kind, C, out_dtype, accumulate, M, N, K);
  if (rc != FP8FG_OK) return rc;
  NoallocDevice* d = nullptr;
  rc = noalloc_device(&d);
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
