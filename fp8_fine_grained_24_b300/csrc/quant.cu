// Fine-grained E4M3 quantizers (DeepSeek-V3 report excerpt, "Fine-Grained
// Quantization"; DeepGEMM article, "Fine-grained scaling"):
//   quant_1x128   one scale per row per 128 columns (activations),
//   quant_128x128 one scale per 128x128 block (weights),
//   requant_128x1 1x128 -> 128x1 retile for the backward pass, written
//                 transposed (channel-major).
//
// All three are the same persistent pipeline. One CTA per SM; warp 0 is a
// TMA producer that streams the input in 16-64 KB chunks (one 128-column
// strip of rows, one 128x128 block, one 128x128 tile) through a ring of
// shared-memory stages; 16 consumer warps read a chunk from shared memory
// into registers, release the stage, reduce the amax (warp shuffles, and for
// the 2-D tiles partial maxima exchanged through shared memory behind an
// mbarrier), then write E4M3 codes and scales straight to global memory
// with row-contiguous stores. The ring keeps about 192 KB of loads in
// flight per SM, so HBM streams continuously while the consumers compute.
//
// The consumers are bound by instruction issue, so the element arithmetic
// is kept lean: values are unpacked already negated (free for BF16) so that
// the correctly rounded quotient runs as five packed f32x2 operations per
// pair (quot2_fma), chunk coordinates advance as a mixed-radix counter
// instead of being divided out per chunk, and the quotient path (exact
// multiply for power-of-two scales, FMA-corrected otherwise) is chosen
// once per chunk by a warp vote.
//
// Every wait is bounded (see mbar_wait_sleep); a timeout is recorded in the
// device status word and the CTA winds down after its copies have landed.
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "quant_math.cuh"
#include "tmap.h"

namespace fp8fg {

namespace {

constexpr int kTile = 128;
constexpr int kConsumerWarps = 16;     // the 1x128 and 128x128 quantizers
constexpr int kRingBytes = 192 * 1024;  // per SM

enum : uint32_t { kStatusTimeoutQuantProducer = 5, kStatusTimeoutQuantConsumer = 6, kStatusTimeoutQuantDrain = 7 };

struct Pipe {
  uint32_t* status;
  uint64_t wait_limit_ns;
  int debug_skip_fill;
};

// Chunk coordinates (d2, d1, d0) of chunk index c = (d2 * R1 + d1) * R0 + d0,
// advanced by a fixed step (gridDim.x) with carries instead of divisions.
struct Walk {
  int64_t d2;
  int d1, d0;
  int r1, r0;
  int64_t s2;
  int s1, s0;

  __device__ __forceinline__ void init(int64_t c, int64_t step, int radix1, int radix0) {
    r1 = radix1;
    r0 = radix0;
    const int64_t per2 = static_cast<int64_t>(r1) * r0;
    d2 = c / per2;
    const int64_t rem = c - d2 * per2;
    d1 = static_cast<int>(rem / r0);
    d0 = static_cast<int>(rem - static_cast<int64_t>(d1) * r0);
    s2 = step / per2;
    const int64_t srem = step - s2 * per2;
    s1 = static_cast<int>(srem / r0);
    s0 = static_cast<int>(srem - static_cast<int64_t>(s1) * r0);
  }

  __device__ __forceinline__ void advance() {
    d0 += s0;
    int carry = d0 >= r0;
    if (carry) d0 -= r0;
    d1 += s1 + carry;
    carry = d1 >= r1;
    if (carry) d1 -= r1;
    d2 += s2 + carry;
  }
};

// Eight consecutive elements of a row from shared memory, negated, as four
// f32 pairs.
template <bool kF32>
__device__ __forceinline__ void load_neg8(const uint8_t* p, uint64_t (&v)[4]) {
  if constexpr (kF32) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 16);
    v[0] = pk2(-a.x, -a.y);
    v[1] = pk2(-a.z, -a.w);
    v[2] = pk2(-b.x, -b.y);
    v[3] = pk2(-b.z, -b.w);
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    v[0] = neg_bf16x2(w.x);
    v[1] = neg_bf16x2(w.y);
    v[2] = neg_bf16x2(w.z);
    v[3] = neg_bf16x2(w.w);
  }
}

__device__ __forceinline__ float amax4pk(const uint64_t (&v)[4]) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) a = amax_pk(v[i], a);
  return a;
}

__device__ __forceinline__ uint2 codes8(const uint64_t (&v)[4]) {
  return make_uint2(e4m3x4_pk(v[0], v[1]), e4m3x4_pk(v[2], v[3]));
}

// ---------------------------------------------------------------- pipeline
// Shared memory: kStages stages of kStageBytes, then full[S], empty[S] and
// Op::kExchBars exchange barriers (8 bytes each), then the exchange buffer.
template <class Op>
struct Layout {
  static constexpr int kBarOff = Op::kStages * Op::kStageBytes;
  static constexpr int kRedOff = (kBarOff + (2 * Op::kStages + Op::kExchBars) * 8 + 15) / 16 * 16;
  static constexpr int kSmem = kRedOff + Op::kRedBytes;
};

// The pipeline's dynamic shared memory. Stages and the exchange buffer are
// addressed as offsets into this array (not through pointers kept in
// structs), so that every consumer access compiles to a shared-memory load
// rather than a generic one.
extern __shared__ __align__(1024) uint8_t quant_smem[];

// Per-chunk context handed to a consumer.
struct Slot {
  uint32_t st_off;  // the stage: byte offset in quant_smem
  uint32_t full, empty, ph;
  uint32_t red_bar;
  uint32_t red_off;  // the exchange buffer: byte offset in quant_smem
  uint32_t it;       // this CTA's chunk counter (exchange-buffer parity)
};

__device__ __forceinline__ const uint8_t* stage_of(const Slot& sl) { return quant_smem + sl.st_off; }
__device__ __forceinline__ float* red_of(const Slot& sl) { return reinterpret_cast<float*>(quant_smem + sl.red_off); }

// Warp 0 lane 0 fills stages; warps 1..Op::kWarps consume them in the same
// chunk order (chunk c = blockIdx.x + i * gridDim.x). Op::kCtasPerSm CTAs
// share an SM.
template <class Op>
__global__ void __launch_bounds__(32 * (1 + Op::kWarps), Op::kCtasPerSm)
    quant_pipe_kernel(const __grid_constant__ CUtensorMap tm, const typename Op::Args a, const Pipe p) {
  uint8_t* const smem = quant_smem;
  constexpr int S = Op::kStages;
  using L = Layout<Op>;
  const uint32_t base = smem_u32(smem);
  const uint32_t bar0 = base + L::kBarOff;
  const uint32_t red_bar = bar0 + 2 * S * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t chunks = a.chunks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar0 + s * 8, 1);
      mbar_init(bar0 + (S + s) * 8, Op::kWarps);
    }
    for (int i = 0; i < Op::kExchBars; ++i) mbar_init(red_bar + i * 8, Op::kWarps);
    fence_barrier_init();
  }
  __syncthreads();

  Walk w;
  Op::walk_init(a, w, blockIdx.x, gridDim.x);
  uint32_t it = 0, s = 0, ph = 0;
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tm);
      for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x, ++it, w.advance()) {
        if (!mbar_wait_sleep(bar0 + (S + s) * 8, ph ^ 1, p.status, kStatusTimeoutQuantProducer, p.wait_limit_ns))
          break;
        if (static_cast<int>(it) != p.debug_skip_fill)  // test hook: a fill that never lands
          Op::issue(tm, a, w, base + s * Op::kStageBytes, bar0 + s * 8);
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
      // No copy may still be landing in shared memory when the CTA exits:
      // wait (bounded, ignoring the error word) for the last fill of each stage.
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
      for (uint32_t i = first; i < it; ++i) {
        if (static_cast<int>(i) == p.debug_skip_fill) continue;
        if (!mbar_wait_sleep(bar0 + (i % S) * 8, (i / S) & 1, nullptr, 0, p.wait_limit_ns))
          atomicCAS(p.status, 0u, kStatusTimeoutQuantDrain);
      }
    }
    return;
  }

  const int cw = warp - 1;
  typename Op::State state{};
  bool ok = true;
  for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x, ++it, w.advance()) {
    const Slot sl{s * Op::kStageBytes, bar0 + s * 8, bar0 + (S + s) * 8, ph, red_bar, L::kRedOff, it};
    if (!Op::consume(a, p, w, sl, cw, lane, state)) {
      ok = false;
      break;
    }
    if (++s == S) {
      s = 0;
      ph ^= 1;
    }
  }
  if (ok) Op::finish(a, p, cw, lane, state);
}

__device__ __forceinline__ bool wait_full(const Slot& sl, const Pipe& p) {
  return mbar_wait_sleep(sl.full, sl.ph, p.status, kStatusTimeoutQuantConsumer, p.wait_limit_ns);
}

// Release a stage once the whole warp has read it into registers. The
// reads went through the generic proxy and the producer's next fill writes
// through the async (TMA) proxy, which the mbarrier handshake alone does not
// order: without the proxy fence a read still in flight could see the next
// chunk (observed on FP32 inputs). Callers also release only after the
// loaded values have been consumed (the amax reduction), so the fence has
// nothing left to wait for.
__device__ __forceinline__ void release(const Slot& sl, int lane) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  if (lane == 0) mbar_arrive(sl.empty);
}

// Post this warp's partial maxima (written before the call) and wait until
// all 16 consumer warps have posted theirs for this chunk.
__device__ __forceinline__ bool exchange(const Slot& sl, const Pipe& p, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(sl.red_bar);
  return mbar_wait_sleep(sl.red_bar, sl.it & 1, p.status, kStatusTimeoutQuantConsumer, p.wait_limit_ns);
}

// ------------------------------------------------------------ 1x128
// Chunk: rows [rb*R, rb*R + R) x columns [kb*128, kb*128 + 128), R = 128
// (BF16) or 64 (FP32), one 32 KB TMA box; kb runs fastest. Consumer warp w
// takes 2*I rows (I = R/32); each half-warp one row per step (16 lanes x 8
// elements), so a warp reads 2 rows per shared-memory instruction and writes
// two 128-byte row segments of q. The scalar work of a tile (the division
// by 448, the reciprocal) is done once per tile rather than on each of its
// 16 lanes: the warp's 2*I row maxima are gathered one per lane, every lane
// computes one scale, and each step fetches its tile's scale by shuffle.
template <bool kF32>
struct Quant1x128 {
  static constexpr int kEsz = kF32 ? 4 : 2;
  static constexpr int kRows = kF32 ? 64 : 128;
  static constexpr int kStageBytes = kRows * kTile * kEsz;
  static constexpr int kWarps = kConsumerWarps, kCtasPerSm = 1;
  static constexpr int kStages = kRingBytes / kStageBytes;
  static constexpr int kRedBytes = 0;
  static constexpr int kExchBars = 0;
  static constexpr int kIters = kRows / kConsumerWarps / 2;  // 4 (BF16) or 2 (FP32)
  struct State {};
  static constexpr int kWarpRows = 2 * kIters;

  struct Args {
    int64_t chunks, M, K, lds;
    int KB;
    uint8_t* q;
    float* s;
    int pow2;
  };

  // d2 = row block, d0 = 128-column block
  static __device__ __forceinline__ void walk_init(const Args& a, Walk& w, int64_t c, int64_t step) {
    w.init(c, step, 1, a.KB);
  }

  static __device__ __forceinline__ void issue(const CUtensorMap& tm, const Args&, const Walk& w, uint32_t dst,
                                               uint32_t full) {
    mbar_arrive_expect_tx(full, kStageBytes);
    tma_load_3d(dst, &tm, full, w.d0 * kTile, static_cast<int32_t>(w.d2 * kRows), 0);
  }

  static __device__ __forceinline__ void finish(const Args&, const Pipe&, int, int, State&) {}

  static __device__ __forceinline__ bool consume(const Args& a, const Pipe& p, const Walk& w, const Slot& sl,
                                                 int cw, int lane, State&) {
    const int half = lane >> 4, j = lane & 15;
    if (!wait_full(sl, p)) return false;
    uint64_t v[kIters][4];
#pragma unroll
    for (int i = 0; i < kIters; ++i)
      load_neg8<kF32>(stage_of(sl) + ((cw * kWarpRows + 2 * i + half) * kTile + j * 8) * kEsz, v[i]);
    // row maxima: after the xor-shuffles every lane of half h holds am[i] of row 2i+h
    float am[kIters];
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      am[i] = amax4pk(v[i]);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) am[i] = fmaxf(am[i], __shfl_xor_sync(0xffffffffu, am[i], o));
    }
    release(sl, lane);
    // lane L takes row t = L % (2I): am[t/2] of half t%2
    const int t = lane & (kWarpRows - 1);
    float my_am = 0.0f;
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const float x = __shfl_sync(0xffffffffu, am[i], 16 * (t & 1));
      if ((t >> 1) == i) my_am = x;
    }
    const float my_s = tile_scale(my_am, a.pow2 != 0);
    const float my_r = __frcp_rn(my_s);
    const int path = warp_quot_mode(make_tile_div_mode(my_s));
    const int64_t row0 = w.d2 * kRows + cw * kWarpRows;
    const int64_t col = static_cast<int64_t>(w.d0) * kTile;
    if (lane < kWarpRows && row0 + lane < a.M) a.s[w.d0 * a.lds + row0 + lane] = my_s;
    uint8_t* qp = a.q + (row0 + half) * a.K + col + j * 8;
    const int64_t rows_left = a.M - row0 - half;
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const float sc = __shfl_sync(0xffffffffu, my_s, 2 * i + half);
      const float rc = __shfl_sync(0xffffffffu, my_r, 2 * i + half);
      quot2_n<4>(v[i], path, sc, rc);
      if (2 * i < rows_left) *reinterpret_cast<uint2*>(qp) = codes8(v[i]);
      qp += 2 * a.K;
    }
    return true;
  }
};

// ------------------------------------------------------------ 128x128
// Chunk: one 128x128 block (32 KB BF16 box; FP32 as two 64-row boxes),
// k blocks fastest. Consumer warp w holds rows 8w .. 8w+7 in registers
// (half-warp per row), reduces its amax, posts it to the exchange buffer and
// arrives on the exchange barrier; after the barrier every warp has the
// block's amax. The buffer is double-buffered by chunk parity: a warp can
// only be one chunk ahead of the slowest, because the barrier needs all 16
// arrivals.
template <bool kF32>
struct Quant128x128 {
  static constexpr int kEsz = kF32 ? 4 : 2;
  static constexpr int kStageBytes = kTile * kTile * kEsz;
  static constexpr int kBoxRows = kF32 ? 64 : 128;
  static constexpr int kWarps = kConsumerWarps, kCtasPerSm = 1;
  static constexpr int kStages = kRingBytes / kStageBytes;
  static constexpr int kRedBytes = 2 * kConsumerWarps * 4;
  static constexpr int kExchBars = 1;
  static constexpr int kIters = kTile / kConsumerWarps / 2;
  struct State {};

  struct Args {
    int64_t chunks, N, K;
    int NB, KB;
    uint8_t* q;
    float* s;
    int pow2;
  };

  // d2 = group, d1 = 128-row block, d0 = 128-column block
  static __device__ __forceinline__ void walk_init(const Args& a, Walk& w, int64_t c, int64_t step) {
    w.init(c, step, a.NB, a.KB);
  }

  static __device__ __forceinline__ void issue(const CUtensorMap& tm, const Args&, const Walk& w, uint32_t dst,
                                               uint32_t full) {
    mbar_arrive_expect_tx(full, kStageBytes);
#pragma unroll
    for (int i = 0; i < kTile / kBoxRows; ++i)
      tma_load_3d(dst + i * kBoxRows * kTile * kEsz, &tm, full, w.d0 * kTile, w.d1 * kTile + i * kBoxRows,
                  static_cast<int32_t>(w.d2));
  }

  static __device__ __forceinline__ void finish(const Args&, const Pipe&, int, int, State&) {}

  static __device__ __forceinline__ bool consume(const Args& a, const Pipe& p, const Walk& w, const Slot& sl,
                                                 int cw, int lane, State&) {
    const int half = lane >> 4, j = lane & 15;
    if (!wait_full(sl, p)) return false;
    uint64_t v[kIters][4];
#pragma unroll
    for (int i = 0; i < kIters; ++i)
      load_neg8<kF32>(stage_of(sl) + ((cw * (2 * kIters) + 2 * i + half) * kTile + j * 8) * kEsz, v[i]);
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < kIters; ++i) am = fmaxf(am, amax4pk(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    release(sl, lane);
    float* rb = red_of(sl) + (sl.it & 1) * kConsumerWarps;
    if (lane == 0) rb[cw] = am;
    if (!exchange(sl, p, lane)) return false;
    const float4* r4 = reinterpret_cast<const float4*>(rb);
#pragma unroll
    for (int i = 0; i < kConsumerWarps / 4; ++i) {
      const float4 t = r4[i];
      am = fmaxf(am, fmaxf(fmaxf(t.x, t.y), fmaxf(t.z, t.w)));
    }
    const float sc = tile_scale(am, a.pow2 != 0);
    const float rc = __frcp_rn(sc);
    const int path = make_tile_div_mode(sc);  // the same block scale in every lane
    const int row_in = w.d1 * kTile + cw * (2 * kIters) + half;
    uint8_t* qp = a.q + (w.d2 * a.N + row_in) * a.K + static_cast<int64_t>(w.d0) * kTile + j * 8;
    const int64_t rows_left = a.N - row_in;
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      quot2_n<4>(v[i], path, sc, rc);
      if (2 * i < rows_left) *reinterpret_cast<uint2*>(qp) = codes8(v[i]);
      qp += 2 * a.K;
    }
    if (cw == 0 && lane == 0) a.s[(w.d2 * a.NB + w.d1) * a.KB + w.d0] = sc;
    return true;
  }
};

// ------------------------------------------------------------ 128x1
// Chunk: one 128-token x 64-channel source tile (E4M3 8 KB plus the 128
// token scales of its 128-channel block, BF16 16 KB, FP32 32 KB), token
// blocks fastest so that consecutive chunks extend the same output rows.
// Two CTAs of 8 consumer warps share an SM, each with half the ring, so two
// tiles' latency chains overlap. Consumer warp w takes tokens 16w .. 16w+15,
// two adjacent channels per lane: per token one shared-memory read covers
// the tile's 64 contiguous channels.
// Two phases per tile, pipelined across tiles so that the cross-warp wait
// of one tile overlaps the reads of the next:
//   A(i): read the tile, reduce this warp's per-channel maxima over its 16
//         tokens, post them to exchange slot i % 4 and arrive on its barrier;
//   B(i): read the tile again (the stage is still held), wait until all 8
//         warps have posted tile i, reduce the 8 partials of each channel,
//         compute the 128x1 scales, quantize, write each channel's 16 codes
//         as one 16-byte store into the transposed output row, and release
//         the stage.
// A warp runs A(i+1) before B(i). Four exchange slots make the reuse safe:
// a warp can only post tile i+4 after B(i+2), which needs every warp's
// A(i+2), which each warp runs after its B(i).
// A tile wholly at or beyond the group's valid rows is not loaded: it
// quantizes to zeros with scale 1.
template <int kSrc>  // 0: E4M3 + 1x128 scales, 1: BF16, 2: FP32
struct Requant128x1 {
  static constexpr int kCh = 64;  // channels per tile
  static constexpr int kWarps = 8, kCtasPerSm = 2;
  static constexpr int kEsz = kSrc == 0 ? 1 : (kSrc == 1 ? 2 : 4);
  static constexpr int kTileBytes = kTile * kCh * kEsz;
  // an E4M3 tile carries the 128 token scales (512 B) of its channel block
  static constexpr int kStageBytes = kTileBytes + (kSrc == 0 ? kTile * 4 : 0);
  static constexpr int kStages = kRingBytes / kCtasPerSm / kStageBytes;
  static constexpr int kSlots = 4;
  static constexpr int kExchBars = kSlots;
  static constexpr int kRedBytes = kSlots * kWarps * kCh * 4;
  // rows past the valid count are +0; stored negated that is (-0, -0)
  static constexpr uint64_t kNegZero2 = 0x8000000080000000ull;

  struct Args {
    int64_t chunks, T, C, ld_t, ld_c;
    int TB, CB;  // 128-token blocks, 64-channel blocks
    const float* s_src;
    const int32_t* valid_rows;
    uint8_t* qT;
    float* sT;
    int pow2;
  };

  // the tile of phase A waiting for its phase B
  struct State {
    bool has;
    Slot sl;
    int64_t g;
    int cb, tb;
  };

  // d2 = group, d1 = 64-channel block, d0 = 128-token block
  static __device__ __forceinline__ void walk_init(const Args& a, Walk& w, int64_t c, int64_t step) {
    w.init(c, step, a.CB, a.TB);
  }

  static __device__ __forceinline__ int64_t valid_of(const Args& a, int64_t g) {
    return a.valid_rows ? static_cast<int64_t>(__ldg(a.valid_rows + g)) : a.T;
  }

  static __device__ __forceinline__ void issue(const CUtensorMap& tm, const Args& a, const Walk& w, uint32_t dst,
                                               uint32_t full) {
    if (static_cast<int64_t>(w.d0) * kTile >= valid_of(a, w.d2)) {
      mbar_arrive(full);  // nothing to load: the consumers write zeros
      return;
    }
    mbar_arrive_expect_tx(full, kStageBytes);
    tma_load_3d(dst, &tm, full, w.d1 * kCh, w.d0 * kTile, static_cast<int32_t>(w.d2));
    if constexpr (kSrc == 0)
      bulk_load(dst + kTileBytes,
                a.s_src + (w.d2 * (a.CB / 2) + w.d1 / 2) * a.ld_t + static_cast<int64_t>(w.d0) * kTile, kTile * 4,
                full);
  }

  // This lane's 16 tokens x 2 channels, negated, as f32 pairs (token k of
  // the warp's group in x[k]); rows past `valid` read as +0.
  static __device__ __forceinline__ void load_tile(const uint8_t* st, int tg, int c0, int64_t t0, int64_t valid,
                                                   uint64_t (&x)[16]) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int t = tg * 16 + k;
      if constexpr (kSrc == 0) {
        const uint32_t b = *reinterpret_cast<const uint16_t*>(st + t * kCh + c0);
        const float2 f = e4m3x2_to_f32(b);
        const float nts = -reinterpret_cast<const float*>(st + kTileBytes)[t];  // token scale, negated
        x[k] = mul2(pk2(f.x, f.y), pk2(nts, nts));
      } else if constexpr (kSrc == 1) {
        x[k] = neg_bf16x2(*reinterpret_cast<const uint32_t*>(st + (t * kCh + c0) * 2));
      } else {
        const float2 f = *reinterpret_cast<const float2*>(st + (t * kCh + c0) * 4);
        x[k] = pk2(-f.x, -f.y);
      }
    }
    if (t0 + 16 > valid) {  // the tile straddles the group's last valid row
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (t0 + k >= valid) x[k] = kNegZero2;
    }
  }

  static __device__ __forceinline__ bool phase_a(const Args& a, const Pipe& p, int64_t g, int tb, const Slot& sl,
                                                 int cw, int lane) {
    const int tg = cw, c0 = 2 * lane;
    const int64_t tile_t0 = static_cast<int64_t>(tb) * kTile;
    const int64_t valid = valid_of(a, g);
    if (!wait_full(sl, p)) return false;
    float a0 = 0.0f, a1 = 0.0f;
    if (tile_t0 < valid) {
      uint64_t x[16];
      load_tile(stage_of(sl), tg, c0, tile_t0 + tg * 16, valid, x);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float2 f = unpk2(x[k]);
        a0 = fmaxf(a0, fabsf(f.x));
        a1 = fmaxf(a1, fabsf(f.y));
      }
    }
    float* rb = red_of(sl) + (sl.it % kSlots) * kWarps * kCh;
    *reinterpret_cast<float2*>(rb + tg * kCh + c0) = make_float2(a0, a1);
    __syncwarp();
    if (lane == 0) mbar_arrive(sl.red_bar + (sl.it % kSlots) * 8);
    return true;
  }

  static __device__ __forceinline__ bool phase_b(const Args& a, const Pipe& p, int64_t g, int cb, int tb,
                                                 const Slot& sl, int cw, int lane) {
    const int tg = cw, c0 = 2 * lane;
    const int64_t tile_t0 = static_cast<int64_t>(tb) * kTile;
    const int64_t t0 = tile_t0 + tg * 16;
    const int64_t valid = valid_of(a, g);
    // read the tile again first: its latency overlaps the exchange wait
    uint64_t x[16];
    if (tile_t0 < valid) {
      load_tile(stage_of(sl), tg, c0, t0, valid, x);
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) x[k] = kNegZero2;
    }
    if (!mbar_wait_sleep(sl.red_bar + (sl.it % kSlots) * 8, (sl.it / kSlots) & 1, p.status,
                         kStatusTimeoutQuantConsumer, p.wait_limit_ns))
      return false;
    release(sl, lane);
    const float* rb = red_of(sl) + (sl.it % kSlots) * kWarps * kCh;
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
      const float2 t = *reinterpret_cast<const float2*>(rb + i * kCh + c0);
      a0 = fmaxf(a0, t.x);
      a1 = fmaxf(a1, t.y);
    }
    const float s0 = tile_scale(a0, a.pow2 != 0), s1 = tile_scale(a1, a.pow2 != 0);
    const int64_t ch = static_cast<int64_t>(cb) * kCh + c0;  // channel index within the group
    if (tg == 0) {
      float* sr = a.sT + (g * a.TB + tb) * a.ld_c + ch;
      sr[0] = s0;
      sr[1] = s1;
    }
    const int m0 = make_tile_div_mode(s0), m1 = make_tile_div_mode(s1);
    const int path = warp_quot_mode(m0 == kQuotDiv || m1 == kQuotDiv ? kQuotDiv
                                    : (m0 == kQuotMul && m1 == kQuotMul ? kQuotMul : kQuotFma));
    // per-lane scale pair (channel c0 in the low half, c0+1 in the high half)
    const float r0 = __frcp_rn(s0), r1 = __frcp_rn(s1);
    if (path == kQuotMul) {
      const uint64_t nr2 = pk2(-r0, -r1);
#pragma unroll
      for (int k = 0; k < 16; ++k) x[k] = mul2(x[k], nr2);
    } else if (path == kQuotFma) {
      const uint64_t s2 = pk2(s0, s1), nr2 = pk2(-r0, -r1);
#pragma unroll
      for (int k = 0; k < 16; ++k) x[k] = quot2_fma(x[k], s2, nr2);
    } else {
      const TileDiv d0{s0, r0, m0}, d1{s1, r1, m1};
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float2 f = unpk2(x[k]);
        x[k] = pk2(tile_quot(-f.x, d0), tile_quot(-f.y, d1));
      }
    }
    // x[k] holds (channel c0, channel c0+1) of token k; gather each channel's
    // 16 tokens into one 16-byte row segment
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4)
      e4m3_transpose4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3], lo[k4], hi[k4]);
    uint8_t* row0 = a.qT + (g * a.C + ch) * a.T + t0;
    *reinterpret_cast<uint4*>(row0) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(row0 + a.T) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    return true;
  }

  static __device__ __forceinline__ bool consume(const Args& a, const Pipe& p, const Walk& w, const Slot& sl,
                                                 int cw, int lane, State& st) {
    if (!phase_a(a, p, w.d2, w.d0, sl, cw, lane)) return false;
    if (st.has && !phase_b(a, p, st.g, st.cb, st.tb, st.sl, cw, lane)) return false;
    st.has = true;
    st.sl = sl;
    st.g = w.d2;
    st.cb = w.d1;
    st.tb = w.d0;
    return true;
  }

  static __device__ __forceinline__ void finish(const Args& a, const Pipe& p, int cw, int lane, State& st) {
    if (st.has) phase_b(a, p, st.g, st.cb, st.tb, st.sl, cw, lane);
  }
};

// ---------------------------------------------------------------- host side
// Raise the kernel's dynamic shared-memory limit once per device.
template <class Op>
cudaError_t ensure_attr() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(quant_pipe_kernel<Op>, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<Op>::kSmem);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

template <class Op>
cudaError_t launch_pipe(const CUtensorMap& tm, const typename Op::Args& a, const Pipe& p, int num_sms,
                        cudaStream_t stream) {
  static_assert(Layout<Op>::kSmem <= 227 * 1024, "shared memory budget");
  cudaError_t e = ensure_attr<Op>();
  if (e != cudaSuccess) return e;
  const int64_t ctas = static_cast<int64_t>(num_sms) * Op::kCtasPerSm;
  const int64_t grid = a.chunks < ctas ? a.chunks : ctas;
  quant_pipe_kernel<Op><<<static_cast<unsigned>(grid), 32 * (1 + Op::kWarps), Layout<Op>::kSmem, stream>>>(tm, a, p);
  return cudaGetLastError();
}

CUtensorMapDataType map_type(int esz) {
  return esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                  : (esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

constexpr int64_t kMaxBlocks = (1ll << 31) - 1;  // block coordinates are 32-bit in the walk

}  // namespace

cudaError_t launch_quant_1x128(const void* x, bool f32, int64_t M, int64_t K, int64_t ldx, uint8_t* q, float* s,
                               int64_t lds, int pow2, const QuantLaunch& l, cudaStream_t stream) {
  const int esz = f32 ? 4 : 2;
  const int rows = f32 ? Quant1x128<true>::kRows : Quant1x128<false>::kRows;
  if (K / kTile > kMaxBlocks) return cudaErrorInvalidValue;
  CUtensorMap tm;
  if (!make_map(&tm, map_type(esz), x, K, M, 1, ldx * esz, M * ldx * esz, kTile, rows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const Pipe p{l.status, l.wait_limit_ns, l.debug_skip_fill};
  const int KB = static_cast<int>(K / kTile);
  const int64_t chunks = ((M + rows - 1) / rows) * KB;
  if (f32) {
    typename Quant1x128<true>::Args a{chunks, M, K, lds, KB, q, s, pow2};
    return launch_pipe<Quant1x128<true>>(tm, a, p, l.num_sms, stream);
  }
  typename Quant1x128<false>::Args a{chunks, M, K, lds, KB, q, s, pow2};
  return launch_pipe<Quant1x128<false>>(tm, a, p, l.num_sms, stream);
}

cudaError_t launch_quant_128x128(const void* w, bool f32, int64_t G, int64_t N, int64_t K, uint8_t* q, float* s,
                                 int pow2, const QuantLaunch& l, cudaStream_t stream) {
  const int esz = f32 ? 4 : 2;
  const int box_rows = f32 ? Quant128x128<true>::kBoxRows : Quant128x128<false>::kBoxRows;
  const int64_t NB = (N + kTile - 1) / kTile, KB = K / kTile;
  if (N > kMaxBlocks || KB > kMaxBlocks) return cudaErrorInvalidValue;
  CUtensorMap tm;
  if (!make_map(&tm, map_type(esz), w, K, N, G, K * esz, N * K * esz, kTile, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const Pipe p{l.status, l.wait_limit_ns, l.debug_skip_fill};
  if (f32) {
    typename Quant128x128<true>::Args a{G * NB * KB, N, K, static_cast<int>(NB), static_cast<int>(KB), q, s, pow2};
    return launch_pipe<Quant128x128<true>>(tm, a, p, l.num_sms, stream);
  }
  typename Quant128x128<false>::Args a{G * NB * KB, N, K, static_cast<int>(NB), static_cast<int>(KB), q, s, pow2};
  return launch_pipe<Quant128x128<false>>(tm, a, p, l.num_sms, stream);
}

cudaError_t launch_requant_128x1(const void* src, int src_kind, const float* s_src, int64_t ld_t, int64_t G,
                                 int64_t T, int64_t C, const int32_t* valid_rows, uint8_t* qT, float* sT,
                                 int64_t ld_c, int pow2, const QuantLaunch& l, cudaStream_t stream) {
  const int esz = src_kind == 0 ? 1 : (src_kind == 1 ? 2 : 4);
  constexpr int kCh = Requant128x1<0>::kCh;
  const int64_t TB = T / kTile, CB = C / kCh;
  if (TB > kMaxBlocks || CB > kMaxBlocks) return cudaErrorInvalidValue;
  CUtensorMap tm;
  if (!make_map(&tm, map_type(esz), src, C, T, G, C * esz, T * C * esz, kCh, kTile, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const Pipe p{l.status, l.wait_limit_ns, l.debug_skip_fill};
  const int tb = static_cast<int>(TB), cb = static_cast<int>(CB);
  switch (src_kind) {
    case 0: {
      typename Requant128x1<0>::Args a{G * TB * CB, T, C, ld_t, ld_c, tb, cb, s_src, valid_rows, qT, sT, pow2};
      return launch_pipe<Requant128x1<0>>(tm, a, p, l.num_sms, stream);
    }
    case 1: {
      typename Requant128x1<1>::Args a{G * TB * CB, T, C, ld_t, ld_c, tb, cb, nullptr, valid_rows, qT, sT, pow2};
      return launch_pipe<Requant128x1<1>>(tm, a, p, l.num_sms, stream);
    }
    default: {
      typename Requant128x1<2>::Args a{G * TB * CB, T, C, ld_t, ld_c, tb, cb, nullptr, valid_rows, qT, sT, pow2};
      return launch_pipe<Requant128x1<2>>(tm, a, p, l.num_sms, stream);
    }
  }
}

}  // namespace fp8fg
