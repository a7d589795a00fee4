// Fine-grained E4M3 quantizers (DeepSeek-V3 report excerpt, pages 1-2):
//   quant_1x128   one scale per row per 128 columns (activations),
//   quant_128x128 one scale per 128x128 block (weights),
//   requant_128x1 1x128 -> 128x1 retile for the backward pass, written
//                 transposed (channel-major).
// All three stream HBM once: 16-byte vector loads and stores, warp-shuffle
// amax reductions, an IEEE division for each tile's scale and a correctly
// rounded quotient x/s per element (tile_quot).
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace fp8fg {

namespace {

constexpr int kTile = 128;

// Eight consecutive input elements kept in their storage format (BF16
// stays packed: 4 registers per 8 values) until they are needed as floats.
template <bool kF32>
struct Raw8;

template <>
struct Raw8<false> {
  uint4 w;
  __device__ __forceinline__ void load(const void* p) { w = __ldcs(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ void zero() { w = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
    v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
    v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
  }
};

template <>
struct Raw8<true> {
  float4 a, b;
  __device__ __forceinline__ void load(const void* p) {
    a = __ldcs(reinterpret_cast<const float4*>(p));
    b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

template <bool kF32>
__device__ __forceinline__ void load8(const void* p, float (&v)[8]) {
  Raw8<kF32> r;
  r.load(p);
  r.get(v);
}

__device__ __forceinline__ float amax8(const float (&v)[8]) {
  float a = fabsf(v[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
  return a;
}

template <bool kF32>
__device__ __forceinline__ float amax8(const Raw8<kF32>& r) {
  float v[8];
  r.get(v);
  return amax8(v);
}

__device__ __forceinline__ uint2 quant8(const float (&v)[8], const TileDiv& d) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = e4m3x2(tile_quot(v[2 * i], d), tile_quot(v[2 * i + 1], d));
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

template <bool kF32>
__device__ __forceinline__ uint2 quant8(const Raw8<kF32>& r, const TileDiv& d) {
  float v[8];
  r.get(v);
  return quant8(v, d);
}

// ------------------------------------------------------------ 1x128
// A half-warp owns one 1x128 tile: 16 lanes x 8 elements. A warp's work unit
// is one row and a run of 2*kUnroll consecutive tiles of it (the two
// half-warps take alternate tiles), so each thread keeps kUnroll 16-byte
// loads in flight and consecutive half-warps read consecutive 256/512-byte
// segments of the row. Units are visited row-major; one 32-bit division per
// unit (the launcher checks that the unit count fits 32 bits).
template <bool kF32, int kUnroll>
__global__ void __launch_bounds__(256) quant_1x128_kernel(const void* __restrict__ x, int64_t ldx,
                                                          int64_t M, int64_t K, uint8_t* __restrict__ q,
                                                          float* __restrict__ s, int64_t lds, int pow2) {
  constexpr int kRun = 2 * kUnroll;
  const uint32_t KB = static_cast<uint32_t>(K / kTile);
  const uint32_t runs_per_row = (KB + kRun - 1) / kRun;
  const uint32_t units = static_cast<uint32_t>(M) * runs_per_row;
  const int lane = threadIdx.x & 31;
  const int j = lane & 15;  // 8-element chunk within the tile
  const int half = lane >> 4;
  const uint32_t warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t warps_total = (gridDim.x * blockDim.x) >> 5;
  const size_t esz = kF32 ? 4 : 2;

  for (uint32_t unit = warp_global; unit < units; unit += warps_total) {
    const uint32_t m = unit / runs_per_row;
    const uint32_t kb0 = (unit - m * runs_per_row) * kRun;
    const char* xrow = static_cast<const char*>(x) + (static_cast<int64_t>(m) * ldx + j * 8) * esz;
    Raw8<kF32> v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t kb = kb0 + 2 * u + half;
      if (kb < KB)
        v[u].load(xrow + static_cast<int64_t>(kb) * kTile * esz);
      else
        v[u].zero();
    }
    uint8_t* qrow = q + static_cast<int64_t>(m) * K + j * 8;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t kb = kb0 + 2 * u + half;
      float a = amax8(v[u]);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      const float sc = tile_scale(a, pow2 != 0);
      if (kb < KB) {
        *reinterpret_cast<uint2*>(qrow + static_cast<int64_t>(kb) * kTile) = quant8(v[u], make_tile_div(sc));
        if (j == 0) s[static_cast<int64_t>(kb) * lds + m] = sc;
      }
    }
  }
}

// ------------------------------------------------------------ 128x128
// One CTA (256 threads) per 128x128 block, held in registers in storage
// format (BF16: 32 registers per thread). Warp w covers rows w*16 .. w*16+15,
// two rows per load instruction (16 lanes x 16 bytes per BF16 row).
template <bool kF32>
__global__ void __launch_bounds__(256) quant_128x128_kernel(const void* __restrict__ w, int64_t N, int64_t K,
                                                            uint8_t* __restrict__ q, float* __restrict__ s,
                                                            int pow2) {
  const int64_t KB = K / kTile;
  const int64_t NB = (N + kTile - 1) / kTile;
  const int64_t blk = blockIdx.x;
  const int64_t g = blk / (NB * KB);
  const int64_t r = blk - g * NB * KB;
  const int64_t nb = r / KB, kb = r - (r / KB) * KB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = lane & 15;
  const size_t esz = kF32 ? 4 : 2;
  const char* wg = static_cast<const char*>(w) + g * N * K * esz;

  constexpr int kRowsPerThread = 8;
  Raw8<kF32> v[kRowsPerThread];
#pragma unroll
  for (int i = 0; i < kRowsPerThread; ++i) {
    const int64_t row = nb * kTile + warp * 16 + i * 2 + (lane >> 4);
    if (row < N)
      v[i].load(wg + (row * K + kb * kTile + chunk * 8) * esz);
    else
      v[i].zero();
  }
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < kRowsPerThread; ++i) a = fmaxf(a, amax8(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  __shared__ float red[8];
  if (lane == 0) red[warp] = a;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
  const float sc = tile_scale(a, pow2 != 0);
  const TileDiv d = make_tile_div(sc);
  uint8_t* qg = q + g * N * K;
#pragma unroll
  for (int i = 0; i < kRowsPerThread; ++i) {
    const int64_t row = nb * kTile + warp * 16 + i * 2 + (lane >> 4);
    if (row < N) {
      *reinterpret_cast<uint2*>(qg + row * K + kb * kTile + chunk * 8) = quant8(v[i], d);
    }
  }
  if (threadIdx.x == 0) s[(g * NB + nb) * KB + kb] = sc;
}

// ------------------------------------------------------------ 128x1
// One CTA per (group, 128-token block, 128-channel block). The source tile
// is dequantized into shared memory as FP32 [token][channel] (row stride 129
// floats: column reads are bank-conflict free), per-channel amax over the
// 128 tokens gives the 128x1 scales, and each output row (one channel, 128
// tokens) is written as eight 16-byte stores.
constexpr int kRqStride = kTile + 1;
constexpr int kRqSmem = kTile * kRqStride * 4 + 2 * kTile * 4;

template <int kSrc>  // 0: E4M3 + 1x128 scales, 1: BF16, 2: FP32
__global__ void __launch_bounds__(256) requant_128x1_kernel(const void* __restrict__ src,
                                                            const float* __restrict__ s_src, int64_t ld_t,
                                                            int64_t T, int64_t C,
                                                            const int32_t* __restrict__ valid_rows,
                                                            uint8_t* __restrict__ qT, float* __restrict__ sT,
                                                            int64_t ld_c, int pow2) {
  extern __shared__ float rq_smem[];
  float* xs = rq_smem;                      // [128][129]
  float* part = rq_smem + kTile * kRqStride;  // [2][128]
  const int64_t TB = T / kTile, CB = C / kTile;
  const int64_t blk = blockIdx.x;
  const int64_t g = blk / (TB * CB);
  const int64_t r = blk - g * TB * CB;
  const int64_t tb = r / CB, cb = r - (r / CB) * CB;
  const int tid = threadIdx.x;
  const int64_t valid = valid_rows ? static_cast<int64_t>(valid_rows[g]) : T;

  // ---- load + dequantize
  if constexpr (kSrc == 0) {
    const uint8_t* sp = static_cast<const uint8_t*>(src) + g * T * C;
    const float* ss = s_src + g * CB * ld_t + cb * ld_t;  // ss[t]: scale of token t, channel block cb
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * 256;      // 1024 chunks of 16 bytes
      const int t = idx >> 3, c16 = idx & 7;
      const int64_t tok = tb * kTile + t;
      float* dst = xs + t * kRqStride + c16 * 16;
      if (tok < valid) {
        const uint4 w = __ldcs(reinterpret_cast<const uint4*>(sp + tok * C + cb * kTile + c16 * 16));
        const float sc = ss[tok];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int b = 0; b < 16; ++b) {
          const uint8_t byte = static_cast<uint8_t>(ws[b >> 2] >> ((b & 3) * 8));
          dst[b] = __fmul_rn(e4m3_to_f32(byte), sc);
        }
      } else {
#pragma unroll
        for (int b = 0; b < 16; ++b) dst[b] = 0.0f;
      }
    }
  } else {
    constexpr bool kF32 = (kSrc == 2);
    constexpr size_t esz = kF32 ? 4 : 2;
    const char* sp = static_cast<const char*>(src) + g * T * C * esz;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = tid + i * 256;      // 2048 chunks of 8 elements
      const int t = idx >> 4, c8 = idx & 15;
      const int64_t tok = tb * kTile + t;
      float* dst = xs + t * kRqStride + c8 * 8;
      float v[8];
      if (tok < valid) {
        load8<kF32>(sp + (tok * C + cb * kTile + c8 * 8) * esz, v);
      } else {
#pragma unroll
        for (int b = 0; b < 8; ++b) v[b] = 0.0f;
      }
#pragma unroll
      for (int b = 0; b < 8; ++b) dst[b] = v[b];
    }
  }
  __syncthreads();

  // ---- per-channel amax over 128 tokens (two threads per channel)
  {
    const int c = tid & 127, half = tid >> 7;
    float a = 0.0f;
#pragma unroll 8
    for (int t = half * 64; t < half * 64 + 64; ++t) a = fmaxf(a, fabsf(xs[t * kRqStride + c]));
    part[half * kTile + c] = a;
  }
  __syncthreads();
  if (tid < kTile) {
    const float sc = tile_scale(fmaxf(part[tid], part[kTile + tid]), pow2 != 0);
    part[tid] = sc;
    sT[g * TB * ld_c + tb * ld_c + cb * kTile + tid] = sc;
  }
  __syncthreads();

  // ---- quantize and write transposed: lane -> channel, 16 tokens per store
  uint8_t* qg = qT + g * C * T;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = tid + i * 256;  // 1024 = 128 channels x 8 token chunks
    const int c = (idx & 31) + ((idx >> 8) << 5);
    const int t16 = (idx >> 5) & 7;
    const TileDiv d = make_tile_div(part[c]);
    uint32_t w[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float* col = xs + (t16 * 16 + b * 4) * kRqStride + c;
      const uint32_t lo = e4m3x2(tile_quot(col[0], d), tile_quot(col[kRqStride], d));
      const uint32_t hi = e4m3x2(tile_quot(col[2 * kRqStride], d), tile_quot(col[3 * kRqStride], d));
      w[b] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(qg + (cb * kTile + c) * T + tb * kTile + t16 * 16) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

int grid_for(int64_t work_items, int per_block_items, int num_sms, int blocks_per_sm) {
  int64_t want = (work_items + per_block_items - 1) / per_block_items;
  int64_t cap = static_cast<int64_t>(num_sms) * blocks_per_sm;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return static_cast<int>(want);
}

// Raise the requantizer's dynamic shared-memory limit once per device.
template <int kSrc>
cudaError_t ensure_requant_attr() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(requant_128x1_kernel<kSrc>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRqSmem);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

}  // namespace

cudaError_t launch_quant_1x128(const void* x, bool f32, int64_t M, int64_t K, int64_t ldx, uint8_t* q, float* s,
                               int64_t lds, int pow2, int num_sms, cudaStream_t stream) {
  constexpr int kUnroll = 4;
  const int64_t runs = M * ((K / kTile + 2 * kUnroll - 1) / (2 * kUnroll));
  if (runs >= (1ll << 32) || M >= (1ll << 32)) return cudaErrorInvalidValue;
  // 256 threads = 8 warps = 8 work units per pass per block
  const int grid = grid_for(runs, 8, num_sms, 8);
  if (f32)
    quant_1x128_kernel<true, kUnroll><<<grid, 256, 0, stream>>>(x, ldx, M, K, q, s, lds, pow2);
  else
    quant_1x128_kernel<false, kUnroll><<<grid, 256, 0, stream>>>(x, ldx, M, K, q, s, lds, pow2);
  return cudaGetLastError();
}

cudaError_t launch_quant_128x128(const void* w, bool f32, int64_t G, int64_t N, int64_t K, uint8_t* q, float* s,
                                 int pow2, cudaStream_t stream) {
  const int64_t blocks = G * ((N + kTile - 1) / kTile) * (K / kTile);
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  if (f32)
    quant_128x128_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w, N, K, q, s, pow2);
  else
    quant_128x128_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w, N, K, q, s, pow2);
  return cudaGetLastError();
}

cudaError_t launch_requant_128x1(const void* src, int src_kind, const float* s_src, int64_t ld_t, int64_t G,
                                 int64_t T, int64_t C, const int32_t* valid_rows, uint8_t* qT, float* sT,
                                 int64_t ld_c, int pow2, cudaStream_t stream) {
  const int64_t blocks = G * (T / kTile) * (C / kTile);
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const unsigned grid = static_cast<unsigned>(blocks);
  cudaError_t e = cudaSuccess;
  switch (src_kind) {
    case 0:
      e = ensure_requant_attr<0>();
      if (e != cudaSuccess) return e;
      requant_128x1_kernel<0><<<grid, 256, kRqSmem, stream>>>(src, s_src, ld_t, T, C, valid_rows, qT, sT, ld_c, pow2);
      break;
    case 1:
      e = ensure_requant_attr<1>();
      if (e != cudaSuccess) return e;
      requant_128x1_kernel<1><<<grid, 256, kRqSmem, stream>>>(src, s_src, ld_t, T, C, valid_rows, qT, sT, ld_c, pow2);
      break;
    default:
      e = ensure_requant_attr<2>();
      if (e != cudaSuccess) return e;
      requant_128x1_kernel<2><<<grid, 256, kRqSmem, stream>>>(src, s_src, ld_t, T, C, valid_rows, qT, sT, ld_c, pow2);
      break;
  }
  return cudaGetLastError();
}

}  // namespace fp8fg
