// FP8 GEMM with power-of-two fine-grained scales applied inside the tensor
// core (tcgen05.mma kind::mxf8f6f4.block_scale, UE8M0 scale factors).
//
// When both operands carry power-of-two scales per row and 128-wide K block
// (the 128x1 tiles of the backward pass with the report's power-of-2
// scaling factors, DeepSeek-V3 report excerpt, page 2, paragraph 1), a
// scale is exactly an UE8M0 exponent, and the product of scaled operands is
// exact. The tensor core can then apply the scales itself (page 2,
// paragraph 3: the request for MMA with group scaling) and accumulate over
// all of K in TMEM: there is no promotion step on the CUDA cores. The
// result equals the promoted GEMM's up to the order of FP32 additions.
//
// Layout (one CTA per SM, 16 warps):
//   warp 0      TMA producer: A 128x128, B 224x128 (K-major, 128-byte
//               swizzle), the 128 row scales of A and 224 of B, 4 stages;
//   warp 1      MMA issuer: per K block 4 x block-scaled MMA (M 128, N 224,
//               K 32) into one of two 224-column accumulators, the scale
//               factors taken from the stage's slot of a TMEM ring;
//   warps 4-7   scale writers, one per TMEM lane quadrant: per K block they
//               turn the stage's FP32 scales into UE8M0 bytes and store
//               them into the ring slot (every quadrant needs its own copy:
//               the rows of quadrant q read B's scale factors from lanes
//               32q..32q+31);
//   warps 8-15  epilogue: when a tile's accumulator is complete, drain it
//               32 columns at a time through a 4 KB staging area and TMA
//               stores (FP32, reduce-add for C +=), releasing the
//               accumulator after the last TMEM load. With two
//               accumulators the drain overlaps the next tile's MMAs.
// TMEM (512 columns): accumulators at 0 and 224, scale-factor slot s at
// 448 + 16 s (A: 4 columns at +0, B: 7 of 8 columns at +8). A TMEM store of
// N columns starts on a multiple of N, so the slots are 16 columns apart.
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"
#include "launch.h"
#include "tmap.h"

namespace fp8fg {

namespace {

using namespace gemm_detail;

struct BsCfg {
  static constexpr int BN = 224;
  static constexpr int kStages = 4;
  static constexpr int kThreads = 16 * 32;  // 128 registers a thread
  static constexpr int kSfWarp0 = 4, kEpiWarp0 = 8, kEpiWarps = 8;
  static constexpr int kAccCols = BN;
  static constexpr int kSfBase = 2 * kAccCols;  // 448
  static constexpr int kSfA = 4, kSfB = (BN + 31) / 32;  // 4 and 7 columns
  static constexpr int kSfBOff = 8, kSfStride = 16;       // B at +8, slots 16 columns apart
  static_assert(kSfA <= kSfBOff && kSfBOff + 8 <= kSfStride && kSfB <= 8, "scale-factor slot layout");
  static constexpr int kTmemCols = 512;
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = BN * BK;
  static constexpr int kSABytes = BM * 4;
  static constexpr int kSBBytes = BN * 4;
  static constexpr int kEpiBytes = 4096;  // 32 rows x 32 FP32 columns per warp
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffEpi = kOffB + kStages * kBBytes;
  static constexpr int kOffSA = kOffEpi + kEpiWarps * kEpiBytes;
  static constexpr int kOffSB = kOffSA + kStages * kSABytes;
  static constexpr int kOffBar = kOffSB + kStages * kSBBytes;
  // full[S], empty[S], sf_full[S], mma_done[S], acc_full[2], acc_empty[2], drain
  static constexpr int kNumBars = 4 * kStages + 4 + 1;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffTmemSlot + 16 + 1024;
  static_assert(kSfBase + kStages * kSfStride <= kTmemCols, "TMEM budget");
  static_assert(kSmem > 116 * 1024 && kSmem <= 227 * 1024, "one CTA per SM within the shared-memory budget");
  static_assert((kOffB % 1024) == 0 && (kOffEpi % 1024) == 0 && (kBBytes % 1024) == 0, "swizzle alignment");
  static_assert((kOffSB % 16) == 0 && (kSBBytes % 16) == 0, "TMA destinations are 16-byte aligned");
};

// A power-of-two scale as an UE8M0 byte replicated over the 32-bit cell
// (every scale-factor ID reads the same). Zero (rows past the matrix, read
// as zero by TMA) maps to the smallest exponent; anything but +0 or a
// normal power of two sets *bad.
__device__ __forceinline__ uint32_t ue8m0x4(float s, bool& bad) {
  const uint32_t b = __float_as_uint(s);
  bad |= (b & 0x807FFFFFu) != 0;
  return ((b >> 23) & 0xFFu) * 0x01010101u;
}

__global__ void __launch_bounds__(BsCfg::kThreads, 1)
    fp8_gemm_bs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                       const __grid_constant__ CUtensorMap tmC, const KArgs a) {
  using C = BsCfg;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t bar0 = sbase + C::kOffBar;
  auto full_bar = [bar0](uint32_t s) { return bar0 + s * 8; };
  auto empty_bar = [bar0](uint32_t s) { return bar0 + (S + s) * 8; };
  auto sfull_bar = [bar0](uint32_t s) { return bar0 + (2 * S + s) * 8; };
  auto mdone_bar = [bar0](uint32_t s) { return bar0 + (3 * S + s) * 8; };
  auto afull_bar = [bar0](uint32_t b) { return bar0 + (4 * S + b) * 8; };
  auto aempty_bar = [bar0](uint32_t b) { return bar0 + (4 * S + 2 + b) * 8; };
  const uint32_t drain_bar = bar0 + (4 * S + 4) * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSA);
    prefetch_tmap(&tmSB);
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1 + 4);  // the MMAs' commit + the four scale writers
      mbar_init(sfull_bar(s), 4);
      mbar_init(mdone_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(afull_bar(b), 1);
      mbar_init(aempty_bar(b), C::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  grid_dependency_sync();

  const int tiles_m = a.tiles_m;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      constexpr uint32_t tx = C::kABytes + C::kBBytes + C::kSABytes + C::kSBBytes;
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x) {
        const int m0 = (t % tiles_m) * BM, n0 = (t / tiles_m) * C::BN;
        for (int kb = 0; kb < a.KB; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1;
          if (!mbar_wait(empty_bar(s), ph ^ 1, a.status, kStatusTimeoutProducer, a.wait_limit_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), tx);
          if (static_cast<int>(it) == a.debug_skip_fill) continue;  // test hook: never filled
          tma_load_3d(sbase + C::kOffA + s * C::kABytes, &tmA, full_bar(s), kb * BK, m0, 0);
          tma_load_3d(sbase + C::kOffB + s * C::kBBytes, &tmB, full_bar(s), kb * BK, n0, 0);
          tma_load_3d(sbase + C::kOffSA + s * C::kSABytes, &tmSA, full_bar(s), m0, kb, 0);
          tma_load_3d(sbase + C::kOffSB + s * C::kSBBytes, &tmSB, full_bar(s), n0, kb, 0);
        }
      }
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
      for (uint32_t i = first; i < it; ++i) mbar_wait(full_bar(i % S), (i / S) & 1, nullptr, 0, a.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = mxf8_idesc(BM, C::BN);
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x, ++tl) {
        const uint32_t b = tl & 1, aph = (tl >> 1) & 1;
        if (!mbar_wait(aempty_bar(b), aph ^ 1, a.status, kStatusTimeoutMma, a.wait_limit_ns)) break;
        for (int kb = 0; kb < a.KB; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1;
          if (!mbar_wait(full_bar(s), ph, a.status, kStatusTimeoutMma, a.wait_limit_ns) ||
              !mbar_wait(sfull_bar(s), ph, a.status, kStatusTimeoutMma, a.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = kmajor_sw128_desc(sbase + C::kOffA + s * C::kABytes);
          const uint64_t bd = kmajor_sw128_desc(sbase + C::kOffB + s * C::kBBytes);
          const uint32_t d = tmem_base + b * C::kAccCols;
          const uint32_t sfa = tmem_base + C::kSfBase + s * C::kSfStride;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_mxf8_bs(d, ad + 2 * k, bd + 2 * k, idesc, sfa, sfa + C::kSfBOff, (kb > 0 || k > 0) ? 1u : 0u);
          mma_commit(empty_bar(s));  // A and B of the stage consumed
          mma_commit(mdone_bar(s));  // the stage's scale-factor slot may be rewritten
        }
        if (ok) mma_commit(afull_bar(b));
      }
      mma_commit(drain_bar);
      if (!mbar_wait(drain_bar, 0, nullptr, 0, a.wait_limit_ns)) atomicCAS(a.status, 0u, kStatusTimeoutDrain);
    }
  } else if (warp >= C::kSfWarp0 && warp < C::kEpiWarp0) {
    // ------------------------------------------------------------ scale-factor writers
    const int q = warp & 3;  // lanes 32q .. 32q+31; lane r writes rows 32c + r of A and B
    const float* ssa = reinterpret_cast<const float*>(smem + C::kOffSA);
    const float* ssb = reinterpret_cast<const float*>(smem + C::kOffSB);
    const uint32_t lane_bits = static_cast<uint32_t>(q * 32) << 16;
    uint32_t it = 0;
    bool ok = true, bad = false;
    for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x) {
      for (int kb = 0; kb < a.KB; ++kb, ++it) {
        const uint32_t s = it % S, ph = (it / S) & 1;
        // the stage's scales have landed, and the MMAs that last read this
        // scale-factor slot (iteration it - S) have completed
        bool got = mbar_wait(full_bar(s), ph, a.status, kStatusTimeoutEpilogue, a.wait_limit_ns);
        got = got && mbar_wait(mdone_bar(s), ph ^ 1, a.status, kStatusTimeoutEpilogue, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        uint32_t va[4], vb[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) va[c] = ue8m0x4(ssa[s * BM + 32 * c + lane], bad);
#pragma unroll
        for (int c = 0; c < C::kSfB; ++c) vb[c] = ue8m0x4(ssb[s * C::BN + 32 * c + lane], bad);
#pragma unroll
        for (int c = C::kSfB; c < 8; ++c) vb[c] = 0;  // the slot's unused eighth column
        const uint32_t col = tmem_base + lane_bits + C::kSfBase + s * C::kSfStride;
        tmem_st4(col, va);
        tmem_st8(col + C::kSfBOff, vb);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(sfull_bar(s));
          mbar_arrive(empty_bar(s));  // the stage's scales have been read
        }
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(a.status, 0u, kStatusScaleNotPow2);
  } else if (warp >= C::kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int g = (warp - C::kEpiWarp0) >> 2;  // column chunks 0-3 or 4-6 (32 columns each)
    const int c_first = g * 4, c_end = g == 0 ? 4 : (C::BN / 32);
    const uint32_t lane_bits = static_cast<uint32_t>(q * 32) << 16;
    uint8_t* region = smem + C::kOffEpi + (warp - C::kEpiWarp0) * C::kEpiBytes;
    uint32_t tl = 0;
    for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x, ++tl) {
      const int m0 = (t % tiles_m) * BM, n0 = (t / tiles_m) * C::BN;
      const uint32_t b = tl & 1, aph = (tl >> 1) & 1;
      const bool got = mbar_wait(afull_bar(b), aph, a.status, kStatusTimeoutEpilogue, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      for (int c = c_first; c < c_end; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem_base + lane_bits + b * C::kAccCols + 32 * c, r);
        if (c + 1 == c_end) {
          // the last TMEM read of this warp: the accumulator may be reused
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(aempty_bar(b));
        }
        if (lane == 0) bulk_wait_read_all();  // the previous chunk's store has read the staging area
        fence_async_shared();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(region + lane * 128 + ((j ^ (lane & 7)) << 4)) =
              make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
        fence_async_shared();
        __syncwarp();
        if (lane == 0) {
          if (a.accumulate)
            tma_reduce_add_3d(&tmC, smem_u32(region), n0 + 32 * c, m0 + 32 * q, 0);
          else
            tma_store_3d(&tmC, smem_u32(region), n0 + 32 * c, m0 + 32 * q, 0);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

bool encode_bs_maps(const GemmProblem& p, MapSet* m) {
  using C = BsCfg;
  const int64_t KB = p.K / BK;
  bool ok = make_map(&m->a, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.A, p.K, p.rows, 1, p.K, p.rows * p.K, BK, BM,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&m->b, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.B, p.K, p.N, 1, p.K, p.N * p.K, BK, C::BN,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&m->sa, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.sA, p.rows, KB, 1, ld4(p.rows) * 4,
                      KB * ld4(p.rows) * 4, BM, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && make_map(&m->sb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.sB, p.N, KB, 1, ld4(p.N) * 4, KB * ld4(p.N) * 4,
                      C::BN, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && make_map(&m->c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.C, p.N, p.rows, 1, p.N * 4, p.rows * p.N * 4, 32, 32,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  m->q = m->sa;  // unused
  return ok;
}

}  // namespace

bool bs_gemm_eligible(const GemmProblem& p) {
  // power-of-two row scales on both operands, dense layout, FP32 output
  return p.b_scale_pow2 && p.mode == kModeDense && p.b_row && p.out_f32 && !p.b_mn_major && p.q_out == nullptr;
}

cudaError_t launch_gemm_bs(const GemmProblem& p, uint32_t* status, uint64_t wait_limit_ns, int debug_skip_fill,
                           int num_sms, cudaStream_t stream, const char** detail) {
  using C = BsCfg;
  MapKey k;
  std::memset(&k, 0, sizeof(k));
  k.A = p.A; k.B = p.B; k.sA = p.sA; k.sB = p.sB; k.C = p.C;
  k.rows = p.rows; k.N = p.N; k.K = p.K; k.groupsA = 1; k.groupsB = 1; k.groupsC = 1;
  k.kind = -3; k.b_row = 1; k.out_f32 = 1;
  MapSet ms;
  if (!map_cache_find(k, &ms)) {
    if (!encode_bs_maps(p, &ms)) {
      *detail = "cuTensorMapEncodeTiled failed (driver entry point missing or arguments rejected)";
      return cudaErrorInvalidValue;
    }
    map_cache_put(k, ms);
  }
  KArgs a;
  std::memset(&a, 0, sizeof(a));
  a.mode = kModeDense;
  a.KB = static_cast<int>(p.K / BK);
  a.rows = static_cast<int>(p.rows);
  a.N = static_cast<int>(p.N);
  a.K = static_cast<int>(p.K);
  a.tiles_m = static_cast<int>((p.rows + BM - 1) / BM);
  a.tiles_n = static_cast<int>((p.N + C::BN - 1) / C::BN);
  const int64_t nt = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  if (nt > 0x7FFFFFFF) {
    *detail = "too many output tiles";
    return cudaErrorInvalidValue;
  }
  a.num_tiles = static_cast<int>(nt);
  a.accumulate = p.accumulate;
  a.C = p.C;
  a.status = status;
  a.wait_limit_ns = wait_limit_ns;
  a.debug_skip_fill = debug_skip_fill;
  if (a.num_tiles == 0) return cudaSuccess;
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(fp8_gemm_bs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) {
      *detail = "cudaFuncSetAttribute(max dynamic shared memory) failed";
      return e;
    }
    attr_done.fetch_or(bit, std::memory_order_release);
  }
  const int grid = a.num_tiles < num_sms ? a.num_tiles : num_sms;
  e = launch_kernel(fp8_gemm_bs_kernel, dim3(grid), dim3(C::kThreads), C::kSmem, stream, ms.a, ms.b, ms.sa, ms.sb,
                    ms.c, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) *detail = "block-scaled GEMM kernel launch failed";
  return e;
}

}  // namespace fp8fg
