// Measurement of the tensor core's own FP8 accumulation (a study, not part
// of the GEMM path).
//
// The DeepSeek-V3 report excerpt (page 1, paragraph 1; page 2, paragraph 1)
// measured that the H800's FP8 MMA keeps only about 14 bits when it adds
// products into its accumulator, which gave an error near 2% at K=4096, and
// fixed it by promoting partial sums to FP32 registers every 128 K. This
// kernel lets the same question be asked of tcgen05 on sm_103a: it computes
// D[128][N] = A[128][K] * B[N][K]^T from unscaled E4M3 codes with the
// tensor-core accumulator restarted every `interval` K elements (a multiple
// of 32, the K extent of one MMA instruction). Each restarted partial is
// added into FP32 registers with an IEEE add. interval >= K chains every MMA
// into one TMEM accumulator (no promotion); interval = 128 is the GEMM
// path's promotion interval with unit scales; interval = 32 promotes after
// every instruction.
//
// Speed does not matter here: one CTA of 4 warps per 128 output columns,
// one shared-memory stage, every MMA group waited for before the next load.
#include "common.cuh"
#include "kernels.h"
#include "launch.h"
#include "tmap.h"

namespace fp8fg {

namespace {

constexpr int kRows = 128;
constexpr int kCols = 128;
constexpr int kBK = 128;
constexpr int kOffA = 0;
constexpr int kOffB = kRows * kBK;              // 16 KB
constexpr int kOffBar = kOffB + kCols * kBK;    // 32 KB
constexpr int kSmem = kOffBar + 64 + 1024;      // + alignment slack

__global__ void __launch_bounds__(128, 1)
    mma_accum_study_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           float* D, int N, int K, int interval, uint32_t* status, uint64_t limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const uint32_t load_bar = sbase + kOffBar;
  const uint32_t mma_bar = load_bar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 16);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kCols;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    mbar_init(load_bar, 1);
    mbar_init(mma_bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  grid_dependency_sync();

  float acc[kCols];
#pragma unroll
  for (int j = 0; j < kCols; ++j) acc[j] = 0.0f;
  constexpr uint32_t idesc = f8_idesc(kRows, kCols);
  const int steps = K / 32;            // MMA instructions along K
  const int per = interval / 32;       // instructions per accumulator restart
  uint32_t lphase = 0, mphase = 0;
  bool ok = true;
  for (int kb = 0; kb < K / kBK && ok; ++kb) {
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(load_bar, kRows * kBK + kCols * kBK);
      tma_load_3d(sbase + kOffA, &tmA, load_bar, kb * kBK, 0, 0);
      tma_load_3d(sbase + kOffB, &tmB, load_bar, kb * kBK, n0, 0);
    }
    ok = mbar_wait(load_bar, lphase, status, kStatusTimeoutProducer, limit_ns);
    lphase ^= 1;
    if (!__syncthreads_and(ok)) break;
    for (int k = 0; k < kBK / 32; ++k) {
      const int step = kb * (kBK / 32) + k;
      const bool fresh = (step % per) == 0;
      const bool last = ((step + 1) % per) == 0 || step + 1 == steps;
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint64_t ad = kmajor_sw128_desc(sbase + kOffA);
        const uint64_t bd = kmajor_sw128_desc(sbase + kOffB);
        mma_f8f6f4(tmem, ad + 2 * k, bd + 2 * k, idesc, fresh ? 0u : 1u);
        mma_commit(mma_bar);
      }
      // every instruction is waited for: the stage is reloaded after the
      // block, and a restart may read the accumulator right away
      ok = mbar_wait(mma_bar, mphase, status, kStatusTimeoutMma, limit_ns);
      mphase ^= 1;
      if (!__syncthreads_and(ok)) break;
      if (last) {
        tc_fence_after();
        const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll
        for (int ch = 0; ch < kCols / 32; ++ch) {
          uint32_t r[32];
          tmem_ld32(taddr + ch * 32, r);
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[ch * 32 + j] = __fadd_rn(acc[ch * 32 + j], __uint_as_float(r[j]));
        }
        tc_fence_before();
        __syncthreads();  // all reads done before the next instruction restarts the accumulator
      }
    }
  }
  if (ok) {
    float* d = D + static_cast<int64_t>(warp * 32 + lane) * N + n0;
#pragma unroll
    for (int j = 0; j < kCols; j += 4) *reinterpret_cast<float4*>(d + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

}  // namespace

cudaError_t launch_mma_accum_study(const uint8_t* A, const uint8_t* B, float* D, int64_t N, int64_t K,
                                   int64_t interval, uint32_t* status, uint64_t wait_limit_ns, cudaStream_t stream,
                                   const char** detail) {
  CUtensorMap tmA, tmB;
  bool ok = make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, kRows, 1, K, kRows * K, kBK, kRows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, 1, K, N * K, kBK, kCols,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) {
    *detail = "cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess && !attr_done[dev & 63]) {
    e = cudaFuncSetAttribute(mma_accum_study_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess) attr_done[dev & 63] = true;
  }
  if (e != cudaSuccess) {
    *detail = "cudaFuncSetAttribute failed";
    return e;
  }
  e = launch_kernel(mma_accum_study_kernel, dim3(static_cast<unsigned>(N / kCols)), dim3(128), kSmem, stream, tmA,
                    tmB, D, static_cast<int>(N), static_cast<int>(K), static_cast<int>(interval), status,
                    wait_limit_ns);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) *detail = "study kernel launch failed";
  return e;
}

}  // namespace fp8fg
