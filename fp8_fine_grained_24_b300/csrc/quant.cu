// Fine-grained E4M3 quantizers (DeepSeek-V3 report excerpt, "Fine-Grained
// Quantization"; DeepGEMM article, "Fine-grained scaling"):
//   quant_1x128   one scale per row per 128 columns (activations),
//   quant_128x128 one scale per 128x128 block (weights),
//   requant_128x1 1x128 -> 128x1 retile for the backward pass, written
//                 transposed (channel-major).
//
// All three are the same persistent pipeline. One CTA per SM; warp 0 is a
// TMA producer that streams the input in 16-64 KB chunks (128 rows x 128
// columns of activations, one 128x128 weight block, one 128-token x
// 128-channel tile) through a ring of shared-memory stages. 16 consumer
// warps, in two teams of 8 that take alternate chunks (one team of 16 for
// FP32 activations and weights), read a chunk into registers, release the
// stage and reduce the amax: warp shuffles, and for 128x128 blocks per-warp
// maxima exchanged through shared memory behind an mbarrier. They write the
// E4M3 codes and scales with row-contiguous global stores; the transposed
// 128x1 output goes through a swizzled image in shared memory and one TMA
// store per warp. The ring keeps about 200 KB of loads in flight per SM, so
// HBM streams continuously while the consumers compute.
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
#include "launch.h"
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
// advanced by a fixed step (the CTAs, times the teams) with carries instead
// of divisions.
struct Walk {
  int64_t d2;
  int d1, d0;
  int r1, r0;
  int64_t s2;
  int s1, s0;

  // Chunk indices, steps and r1 * r0 are below 2^31 (the launchers check
  // the chunk count), so the divisions run in 32 bits: a 64-bit division is
  // a long software sequence, and the producer's first copy waits for it.
  __device__ __forceinline__ void init(int64_t c, int64_t step, int radix1, int radix0) {
    r1 = radix1;
    r0 = radix0;
    const uint32_t per2 = static_cast<uint32_t>(r1) * static_cast<uint32_t>(r0);
    const uint32_t c32 = static_cast<uint32_t>(c), st32 = static_cast<uint32_t>(step);
    const uint32_t q2 = c32 / per2, rem = c32 - q2 * per2;
    d2 = q2;
    d1 = static_cast<int>(rem / static_cast<uint32_t>(r0));
    d0 = static_cast<int>(rem - static_cast<uint32_t>(d1) * static_cast<uint32_t>(r0));
    const uint32_t t2 = st32 / per2, srem = st32 - t2 * per2;
    s2 = t2;
    s1 = static_cast<int>(srem / static_cast<uint32_t>(r0));
    s0 = static_cast<int>(srem - static_cast<uint32_t>(s1) * static_cast<uint32_t>(r0));
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

// Eight quotients (four pairs) -> eight E4M3 bytes, the first in the low byte.
__device__ __forceinline__ uint2 codes8(const uint64_t (&v)[4]) {
  return make_uint2(e4m3x4_pk(v[0], v[1]), e4m3x4_pk(v[2], v[3]));
}

// ---------------------------------------------------------------- pipeline
// Shared memory: Op::kOutBytes of output staging (1024-byte aligned, for
// swizzled TMA stores), kStages stages of kStageBytes, then full[S],
// empty[S] and Op::kExchBars exchange barriers (8 bytes each), then the
// exchange buffer.
template <class Op>
struct Layout {
  static_assert(Op::kOutBytes % 1024 == 0, "output staging keeps the stages 1024-byte aligned");
  static constexpr int kStageOff = Op::kOutBytes;
  static constexpr int kBarOff = kStageOff + Op::kStages * Op::kStageBytes;
  static constexpr int kRedOff = (kBarOff + (2 * Op::kStages + Op::kExchBars) * 8 + 15) / 16 * 16;
  // + slack to align the output staging to 1024 bytes at run time
  static constexpr int kSmem = kRedOff + Op::kRedBytes + (Op::kOutBytes ? 1024 : 0);
};

// The pipeline's dynamic shared memory. Stages and the exchange buffer are
// addressed as offsets into this array (not through pointers kept in
// structs), so that every consumer access compiles to a shared-memory load
// rather than a generic one.
extern __shared__ __align__(1024) uint8_t quant_smem[];

// Per-chunk context handed to a consumer. Offsets are bytes from quant_smem;
// the layout starts `off` bytes in (1024-byte alignment of the output
// staging, 0 for ops without it).
struct Slot {
  uint32_t off;
  uint32_t st_off;  // the stage
  uint32_t full, empty, ph;
  uint32_t red_bar;
  uint32_t red_off;  // the exchange buffer
  uint32_t it;       // this CTA's chunk counter (exchange-buffer parity)
  const CUtensorMap* tmo;  // output tensor map (ops that store through TMA)
};

__device__ __forceinline__ const uint8_t* stage_of(const Slot& sl) { return quant_smem + sl.st_off; }
__device__ __forceinline__ float* red_of(const Slot& sl) { return reinterpret_cast<float*>(quant_smem + sl.red_off); }

// Warp 0 lane 0 fills stages in chunk order (chunk c = blockIdx.x +
// i * gridDim.x); warps 1..Op::kWarps consume them, in Op::kTeams teams of
// Op::kTeamWarps warps, team t taking chunks i = t mod kTeams. Op::kCtasPerSm
// CTAs share an SM.
template <class Op>
__global__ void __launch_bounds__(32 * (1 + Op::kWarps), Op::kCtasPerSm)
    quant_pipe_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tmo,
                      const typename Op::Args a, const Pipe p) {
  constexpr int S = Op::kStages;
  using L = Layout<Op>;
  const uint32_t raw = smem_u32(quant_smem);
  const uint32_t off = Op::kOutBytes ? ((1024u - (raw & 1023u)) & 1023u) : 0u;
  const uint32_t base = raw + off;
  const uint32_t bar0 = base + L::kBarOff;
  const uint32_t red_bar = bar0 + 2 * S * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t chunks = a.chunks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar0 + s * 8, 1);
      mbar_init(bar0 + (S + s) * 8, Op::kReleasers);
    }
    for (int i = 0; i < Op::kExchBars; ++i) mbar_init(red_bar + i * 8, Op::kTeamWarps);
    fence_barrier_init();
  }
  __syncthreads();
  grid_dependency_sync();

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
          Op::issue(tm, a, w, base + L::kStageOff + s * Op::kStageBytes, bar0 + s * 8);
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
  const int team = Op::kTeams > 1 ? cw / Op::kTeamWarps : 0;
  if (Op::kTeams > 1) {
    Op::walk_init(a, w, static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(team) * gridDim.x,
                  static_cast<int64_t>(Op::kTeams) * gridDim.x);
    it = s = team;
  }
  typename Op::State state{};
  bool ok = true;
  for (int64_t c = blockIdx.x + static_cast<int64_t>(team) * gridDim.x; c < chunks;
       c += static_cast<int64_t>(Op::kTeams) * gridDim.x, it += Op::kTeams, w.advance()) {
    const Slot sl{off, off + L::kStageOff + s * Op::kStageBytes, bar0 + s * 8, bar0 + (S + s) * 8, ph, red_bar,
                  off + L::kRedOff, it, &tmo};
    if (!Op::consume(a, p, w, sl, cw, lane, state)) {
      ok = false;
      break;
    }
    s += Op::kTeams;
    if (s >= S) {
      s -= S;
      ph ^= 1;
    }
  }
  if (ok) Op::finish(a, p, cw, lane, state);
  if (Op::kOutBytes && lane == 0) bulk_wait_all();  // stores issued by this warp
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

// ------------------------------------------------------------ 1x128
// Chunk: rows [rb*R, rb*R + R) x columns [kb*128, kb*128 + 128), R = 128
// (BF16) or 64 (FP32), one 32 KB TMA box; kb runs fastest. A warp takes
// 2*I consecutive rows of the chunk; each half-warp one row per step (16
// lanes x 8 elements), so a warp reads 2 rows per shared-memory instruction
// and writes two 128-byte row segments of q. The scalar work of a tile (the
// division by 448, the reciprocal) is done once per tile rather than on each
// of its 16 lanes: a reduce-scatter of the 2*I row maxima over each half's
// lanes (2I shuffles in all, not 4 per row) leaves every lane one row's
// maximum, every lane computes that row's scale, and each step fetches its
// tile's scale by shuffle.
// BF16: two teams of 8 warps take alternate chunks (I = 8), so that the
// shuffle and scale chains of one chunk overlap another's; a lane keeps
// its rows as raw BF16 words, takes the row maxima on packed pairs and
// unpacks only for the quotient. FP32: one team of 16 warps (I = 2).
template <bool kF32>
struct Quant1x128 {
  static constexpr int kEsz = kF32 ? 4 : 2;
  static constexpr int kRows = kF32 ? 64 : 128;
  static constexpr int kStageBytes = kRows * kTile * kEsz;
  static constexpr int kWarps = kConsumerWarps, kCtasPerSm = 1, kOutBytes = 0;
  static constexpr int kTeams = kF32 ? 1 : 2, kTeamWarps = kWarps / kTeams, kReleasers = kTeamWarps;
  static constexpr int kStages = kRingBytes / kStageBytes;
  static constexpr int kRedBytes = 0;
  static constexpr int kExchBars = 0;
  static constexpr int kIters = kRows / kTeamWarps / 2;  // 8 (BF16) or 2 (FP32)
  static constexpr int kWarpRows = 2 * kIters;
  static_assert(kWarpRows <= 32, "one row maximum per lane");
  struct State {};

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
    const int wt = cw % kTeamWarps;
    const int half = lane >> 4, j = lane & 15;
    if (!wait_full(sl, p)) return false;
    // the lane's 8 elements of row 2i + half, raw (BF16: one 16-byte word;
    // FP32: two)
    constexpr int kWords = kF32 ? 2 : 1;
    uint4 v[kIters][kWords];
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const uint8_t* src = stage_of(sl) + ((wt * kWarpRows + 2 * i + half) * kTile + j * 8) * kEsz;
#pragma unroll
      for (int u = 0; u < kWords; ++u) v[i][u] = *reinterpret_cast<const uint4*>(src + 16 * u);
    }
    // the lane's maxima of its kIters rows (row 2i + half for am[i])
    float am[kIters];
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      if constexpr (kF32) {
        float m = 0.0f;
#pragma unroll
        for (int u = 0; u < 2; ++u)
          m = fmaxf(m, fmaxf(fmaxf(fabsf(__uint_as_float(v[i][u].x)), fabsf(__uint_as_float(v[i][u].y))),
                             fmaxf(fabsf(__uint_as_float(v[i][u].z)), fabsf(__uint_as_float(v[i][u].w)))));
        am[i] = m;
      } else {
        uint32_t m0 = v[i][0].x, m1 = v[i][0].z;
        asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m0) : "r"(v[i][0].y));
        asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m1) : "r"(v[i][0].w));
        asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m0) : "r"(m1));
        am[i] = fmaxf(__uint_as_float((m0 << 16) & 0x7FFFFFFFu), __uint_as_float(m0 & 0x7FFF0000u));
      }
    }
    // Reduce-scatter of the kIters maxima over the 16 lanes of the half:
    // at lane bit 3, 2, ... the lane with the bit clear keeps the first half
    // of its values, its partner the second, each taking the max with what
    // the other sends; the remaining kShift lane bits hold copies of one row
    // and finish with a plain butterfly. Afterwards lane j of the half holds
    // the maximum of row 2 * (j >> kShift) + half.
    constexpr int kLog = kIters == 8 ? 3 : (kIters == 4 ? 2 : (kIters == 2 ? 1 : 0));
    static_assert((1 << kLog) == kIters, "row count per half");
    constexpr int kShift = 4 - kLog;
#pragma unroll
    for (int r = 0; r < kLog; ++r) {
      const int bit = 3 - r, n = kIters >> r;
      const bool upper = (lane >> bit) & 1;
#pragma unroll
      for (int q = 0; q < n / 2; ++q) {
        const float send = upper ? am[q] : am[q + n / 2];
        const float keep = upper ? am[q + n / 2] : am[q];
        am[q] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 1 << bit));
      }
    }
#pragma unroll
    for (int bit = kShift - 1; bit >= 0; --bit) am[0] = fmaxf(am[0], __shfl_xor_sync(0xffffffffu, am[0], 1 << bit));
    release(sl, lane);
    const float my_am = am[0];
    const int my_row = 2 * (j >> kShift) + half;  // of the warp's kWarpRows rows
    const float my_s = tile_scale(my_am, a.pow2 != 0);
    const float my_r = __frcp_rn(my_s);
    const int path = warp_quot_mode(make_tile_div_mode(my_s));
    const int64_t row0 = w.d2 * kRows + wt * kWarpRows;
    const int64_t col = static_cast<int64_t>(w.d0) * kTile;
    if ((j & ((1 << kShift) - 1)) == 0 && row0 + my_row < a.M) a.s[w.d0 * a.lds + row0 + my_row] = my_s;
    uint8_t* qp = a.q + (row0 + half) * a.K + col + j * 8;
    const int64_t rows_left = a.M - row0 - half;
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      // row 2i + half's scale: lane (i << kShift) of this half
      const float sc = __shfl_sync(0xffffffffu, my_s, 16 * half + (i << kShift));
      const float rc = __shfl_sync(0xffffffffu, my_r, 16 * half + (i << kShift));
      uint64_t x[4];
      if constexpr (kF32) {
        x[0] = pk2(-__uint_as_float(v[i][0].x), -__uint_as_float(v[i][0].y));
        x[1] = pk2(-__uint_as_float(v[i][0].z), -__uint_as_float(v[i][0].w));
        x[2] = pk2(-__uint_as_float(v[i][1].x), -__uint_as_float(v[i][1].y));
        x[3] = pk2(-__uint_as_float(v[i][1].z), -__uint_as_float(v[i][1].w));
      } else {
        x[0] = neg_bf16x2(v[i][0].x);
        x[1] = neg_bf16x2(v[i][0].y);
        x[2] = neg_bf16x2(v[i][0].z);
        x[3] = neg_bf16x2(v[i][0].w);
      }
      quot2_n<4>(x, path, sc, rc);
      if (2 * i < rows_left) *reinterpret_cast<uint2*>(qp) = codes8(x);
      qp += 2 * a.K;
    }
    return true;
  }
};

// ------------------------------------------------------------ 128x128
// Chunk: one 128x128 block (32 KB BF16 box; FP32 as two 64-row boxes),
// k blocks fastest. The consumer warps of a team split the block's rows
// (half-warp per row, 16 lanes x 8 elements), reduce their amax, post it to
// the team's exchange buffer and arrive on the team's exchange barrier;
// after the barrier every warp of the team has the block's amax. A team's
// buffer is double-buffered by the parity of the team's chunks: a warp can
// only be one chunk ahead of the slowest of its team, because the barrier
// needs all of the team's arrivals.
// BF16: two teams of 8 warps take alternate blocks, so that one team's
// exchange wait overlaps the other's loads. A warp holds its 16 rows as raw
// BF16 words (32 registers), takes the amax on packed pairs
// (max.xorsign.abs.bf16x2 keeps |a| or |b|, the sign bit is dropped at the
// end) and unpacks only for the quotient. FP32: one team of 16 warps of
// 8 rows each.
template <bool kF32>
struct Quant128x128 {
  static constexpr int kEsz = kF32 ? 4 : 2;
  static constexpr int kStageBytes = kTile * kTile * kEsz;
  static constexpr int kBoxRows = kF32 ? 64 : 128;
  static constexpr int kWarps = kConsumerWarps, kCtasPerSm = 1, kOutBytes = 0;
  static constexpr int kTeams = kF32 ? 1 : 2, kTeamWarps = kWarps / kTeams, kReleasers = kTeamWarps;
  static constexpr int kStages = kRingBytes / kStageBytes;
  static constexpr int kRedBytes = kTeams * 2 * kTeamWarps * 4;
  static constexpr int kExchBars = kTeams;
  static constexpr int kIters = kTile / kTeamWarps / 2;  // row pairs per warp
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

  // max(|x|) over a lane's packed BF16 words
  static __device__ __forceinline__ float bf16_amax(const uint4 (&v)[kIters]) {
    uint32_t m0 = 0, m1 = 0;
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m0) : "r"(v[i].x));
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m1) : "r"(v[i].y));
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m0) : "r"(v[i].z));
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m1) : "r"(v[i].w));
    }
    asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m0) : "r"(m1));
    return fmaxf(__uint_as_float((m0 << 16) & 0x7FFFFFFFu), __uint_as_float(m0 & 0x7FFF0000u));
  }

  static __device__ __forceinline__ bool consume(const Args& a, const Pipe& p, const Walk& w, const Slot& sl,
                                                 int cw, int lane, State&) {
    const int team = cw / kTeamWarps, wt = cw % kTeamWarps;
    const int half = lane >> 4, j = lane & 15;
    const uint32_t tit = sl.it / kTeams;  // this team's chunk counter
    if (!wait_full(sl, p)) return false;
    // FP32: a row's 8 elements are two 16-byte words; the lane keeps both
    // halves of each row pair in consecutive entries
    constexpr int kWords = kF32 ? 2 * kIters : kIters;
    uint4 v[kWords];
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const uint8_t* src = stage_of(sl) + ((wt * (2 * kIters) + 2 * i + half) * kTile + j * 8) * kEsz;
      if constexpr (kF32) {
        v[2 * i] = *reinterpret_cast<const uint4*>(src);
        v[2 * i + 1] = *reinterpret_cast<const uint4*>(src + 16);
      } else {
        v[i] = *reinterpret_cast<const uint4*>(src);
      }
    }
    float am;
    if constexpr (kF32) {
      am = 0.0f;
#pragma unroll
      for (int i = 0; i < kWords; ++i)
        am = fmaxf(am, fmaxf(fmaxf(fabsf(__uint_as_float(v[i].x)), fabsf(__uint_as_float(v[i].y))),
                             fmaxf(fabsf(__uint_as_float(v[i].z)), fabsf(__uint_as_float(v[i].w)))));
    } else {
      am = bf16_amax(v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    release(sl, lane);
    float* rb = red_of(sl) + (team * 2 + (tit & 1)) * kTeamWarps;
    const uint32_t bar = sl.red_bar + team * 8;
    if (lane == 0) rb[wt] = am;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    if (!mbar_wait_sleep(bar, tit & 1, p.status, kStatusTimeoutQuantConsumer, p.wait_limit_ns)) return false;
    const float4* r4 = reinterpret_cast<const float4*>(rb);
#pragma unroll
    for (int i = 0; i < kTeamWarps / 4; ++i) {
      const float4 t = r4[i];
      am = fmaxf(am, fmaxf(fmaxf(t.x, t.y), fmaxf(t.z, t.w)));
    }
    const float sc = tile_scale(am, a.pow2 != 0);
    const float rc = __frcp_rn(sc);
    const int path = make_tile_div_mode(sc);  // the same block scale in every lane
    const int row_in = w.d1 * kTile + wt * (2 * kIters) + half;
    uint8_t* qp = a.q + (w.d2 * a.N + row_in) * a.K + static_cast<int64_t>(w.d0) * kTile + j * 8;
    const int64_t rows_left = a.N - row_in;
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      uint64_t x[4];
      if constexpr (kF32) {
        const uint4 lo = v[2 * i], hi = v[2 * i + 1];
        x[0] = pk2(-__uint_as_float(lo.x), -__uint_as_float(lo.y));
        x[1] = pk2(-__uint_as_float(lo.z), -__uint_as_float(lo.w));
        x[2] = pk2(-__uint_as_float(hi.x), -__uint_as_float(hi.y));
        x[3] = pk2(-__uint_as_float(hi.z), -__uint_as_float(hi.w));
      } else {
        x[0] = neg_bf16x2(v[i].x);
        x[1] = neg_bf16x2(v[i].y);
        x[2] = neg_bf16x2(v[i].z);
        x[3] = neg_bf16x2(v[i].w);
      }
      quot2_n<4>(x, path, sc, rc);
      if (2 * i < rows_left) *reinterpret_cast<uint2*>(qp) = codes8(x);
      qp += 2 * a.K;
    }
    if (wt == 0 && lane == 0) a.s[(w.d2 * a.NB + w.d1) * a.KB + w.d0] = sc;
    return true;
  }
};

// ------------------------------------------------------------ 128x1
// Chunk: one 128-token x 128-channel source tile (E4M3 16 KB plus the 128
// token scales of its channel block, BF16 32 KB, FP32 64 KB), token blocks
// fastest so that consecutive chunks extend the same output rows.
//
// Each consumer warp owns 16 channels of the tile across all 128 tokens, so
// a channel's amax is a reduction inside one warp: no warp waits for
// another, and the values stay in registers from load to store. Lane (m, h)
// (m = lane / 2, h = lane % 2) holds channels 8h .. 8h+7 of the warp's 16
// for tokens 8m .. 8m+7: 64 elements.
//
// Shared-memory layout. The tile arrives through a rank-4 view of the
// source, (32-byte column group, token, group, batch), as
// [group][128 tokens][32 bytes]: a lane's 8 channels of one token are 8, 16
// or 32 contiguous bytes, and consecutive tokens of a group are 32 bytes
// apart, so the four tokens t % 4 = 0..3 of one group cover all banks.
// Lane (m, h) reads its k-th token as 8m + (k ^ (m % 8)): at every read the
// 16 lanes of one h are spread over the four residues (two-way conflicts
// for E4M3 and FP32 rows, none for BF16). The output bytes are permuted
// back (one byte permute per 4 bytes) before the store.
//
// Output: each warp writes its 16 channel rows of the transposed tile
// (16 x 128 codes) into its own 2 KB image in shared memory (128-byte
// swizzled) and sends it with one TMA store; before it rewrites the image
// for its next tile it waits until that store has read it.
//
// Two teams of 8 consumer warps take alternate tiles (one team for FP32,
// whose 64 KB stages leave room for few), so that one team's loads and
// reductions overlap the other's.
//
// A tile wholly at or beyond the group's valid rows is not loaded: it
// quantizes to zeros with scale 1.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t c0, int32_t c1,
                                            int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

template <int kSrc>  // 0: E4M3 + 1x128 scales, 1: BF16, 2: FP32
struct Requant128x1 {
  static constexpr int kEsz = kSrc == 0 ? 1 : (kSrc == 1 ? 2 : 4);
  static constexpr int kTeams = kSrc == 2 ? 1 : 2;
  static constexpr int kTeamWarps = 8;  // 8 x 16 channels
  static constexpr int kWarps = kTeams * kTeamWarps, kCtasPerSm = 1;
  static constexpr int kReleasers = kTeamWarps;  // one team reads each stage
  static constexpr int kRow = 32;                // bytes of a token row in one column group
  static constexpr int kGroupBytes = kTile * kRow;
  static constexpr int kTileBytes = kTile * kTile * kEsz;
  // an E4M3 tile carries its 128 token scales (512 B)
  static constexpr int kStageBytes = kTileBytes + (kSrc == 0 ? kTile * 4 : 0);
  static constexpr int kImageBytes = 16 * kTile;  // a warp's 16 channel rows
  static constexpr int kOutBytes = kWarps * kImageBytes;
  static constexpr int kExchBars = 0, kRedBytes = 0;
  static constexpr int kStages = (227 * 1024 - 1024 - kOutBytes - 512) / kStageBytes;
  static_assert(kStages >= 2 * kTeams, "ring depth");
  // rows past the valid count are +0; stored negated that is (-0, -0)
  static constexpr uint64_t kNegZero2 = 0x8000000080000000ull;

  struct Args {
    int64_t chunks, T, C, ld_t, ld_c;
    int TB, CB;  // 128-token blocks, 128-channel blocks
    const float* s_src;
    const int32_t* valid_rows;
    float* sT;
    int pow2;
  };

  struct State {};

  // d2 = group, d1 = 128-channel block, d0 = 128-token block
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
    tma_load_4d(dst, &tm, full, 0, w.d0 * kTile, w.d1 * (kTile * kEsz / kRow), static_cast<int32_t>(w.d2));
    if constexpr (kSrc == 0)
      bulk_load(dst + kTileBytes, a.s_src + (w.d2 * a.CB + w.d1) * a.ld_t + static_cast<int64_t>(w.d0) * kTile,
                kTile * 4, full);
  }

  // The lane's 8 channels of token t, negated, as 4 f32 pairs.
  static __device__ __forceinline__ void load_token(const uint8_t* src, int t, float ts, uint64_t (&v)[4]) {
    const uint8_t* p = src + t * kRow;
    if constexpr (kSrc == 0) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      const uint64_t ns = pk2(-ts, -ts);
      v[0] = mul2(e4m3x2_lo_pk(w.x), ns);
      v[1] = mul2(e4m3x2_hi_pk(w.x), ns);
      v[2] = mul2(e4m3x2_lo_pk(w.y), ns);
      v[3] = mul2(e4m3x2_hi_pk(w.y), ns);
    } else if constexpr (kSrc == 1) {
      const uint4 w = *reinterpret_cast<const uint4*>(p);
      v[0] = neg_bf16x2(w.x);
      v[1] = neg_bf16x2(w.y);
      v[2] = neg_bf16x2(w.z);
      v[3] = neg_bf16x2(w.w);
    } else {
      const float4 a = *reinterpret_cast<const float4*>(p);
      const float4 b = *reinterpret_cast<const float4*>(p + 16);
      v[0] = pk2(-a.x, -a.y);
      v[1] = pk2(-a.z, -a.w);
      v[2] = pk2(-b.x, -b.y);
      v[3] = pk2(-b.z, -b.w);
    }
  }

  // One step of the reduce-scatter of N channel maxima over lane bit `bit`:
  // the lane with the bit clear keeps the first N/2 channels, its partner
  // the last N/2, each taking the max with what the other sends.
  template <int N>
  static __device__ __forceinline__ void reduce_half(float (&v)[8], int lane, int bit) {
    const bool upper = (lane >> bit) & 1;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float send = upper ? v[i] : v[i + N / 2];
      const float keep = upper ? v[i + N / 2] : v[i];
      v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 1 << bit));
    }
  }

  static __device__ __forceinline__ bool consume(const Args& a, const Pipe& p, const Walk& w, const Slot& sl,
                                                 int cw, int lane, State&) {
    const int wt = cw % kTeamWarps;           // the warp's 16 channels: 16 wt .. 16 wt + 15
    const int m = lane >> 1, h = lane & 1;    // tokens 8m .. 8m+7, channels 8h .. 8h+7
    const int c0 = 16 * wt + 8 * h;           // first channel of the lane in the tile
    const int64_t g = w.d2;
    const int cb = w.d1, tb = w.d0;
    const int64_t nvalid = valid_of(a, g) - static_cast<int64_t>(tb) * kTile;  // valid tokens of the tile

    if (!wait_full(sl, p)) return false;
    const int m7 = m & 7;
    uint64_t x[8][4];  // x[k][j]: token 8m + (k ^ m7), channels c0 + 2j, c0 + 2j + 1 (negated)
    if (nvalid > 0) {
      const uint8_t* src = stage_of(sl) + (c0 * kEsz / kRow) * kGroupBytes + (c0 * kEsz) % kRow + 8 * m * kRow;
      const float* ts = reinterpret_cast<const float*>(stage_of(sl) + kTileBytes) + 8 * m;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int u = k ^ m7;
        load_token(src, u, kSrc == 0 ? ts[u] : 1.0f, x[k]);
      }
      if (nvalid < kTile) {  // the tile straddles the group's last valid row
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (8 * m + (k ^ m7) >= nvalid) {
#pragma unroll
            for (int j = 0; j < 4; ++j) x[k][j] = kNegZero2;
          }
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) x[k][j] = kNegZero2;
    }
    release(sl, lane);

    // amax of each of the lane's 8 channels over its 8 tokens, then over the
    // 16 lanes of the same h: after the reduce-scatter lane (m, h) holds
    // channel c0 + j, j = 4 m3 + 2 m2 + m1 (m = 8 m3 + 4 m2 + 2 m1 + m0).
    float am[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float e = 0.0f, o = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 f = unpk2(x[k][j]);
        e = fmaxf(e, fabsf(f.x));
        o = fmaxf(o, fabsf(f.y));
      }
      am[2 * j] = e;
      am[2 * j + 1] = o;
    }
    reduce_half<8>(am, lane, 4);
    reduce_half<4>(am, lane, 3);
    reduce_half<2>(am, lane, 2);
    am[0] = fmaxf(am[0], __shfl_xor_sync(0xffffffffu, am[0], 2));
    const int jm = 4 * ((m >> 3) & 1) + 2 * ((m >> 2) & 1) + ((m >> 1) & 1);
    const float s = tile_scale(am[0], a.pow2 != 0);
    const float r = __frcp_rn(s);
    if ((m & 1) == 0)
      a.sT[(g * a.TB + tb) * a.ld_c + static_cast<int64_t>(cb) * kTile + c0 + jm] = s;
    const int path = warp_quot_mode(make_tile_div_mode(s));

    // Per channel pair (2j, 2j+1): the scales from the lanes that hold them
    // (channel c0 + i sits in lane h + 2 (8 i2 + 4 i1 + 2 i0), i = 4 i2 +
    // 2 i1 + i0), the quotients, then the codes: channel c0 + i, 8 tokens ->
    // 8 bytes, byte k for token 8m + (k ^ m7); byte permutes put token
    // 8m + p in byte p (p ^ m7 selects it). Image row 8h + i, bytes
    // 8m .. 8m+7 (128-byte swizzle: 16-byte chunk m/2 of row r at chunk
    // (m/2) ^ (r % 8)).
    const uint32_t img = sl.off + cw * kImageBytes;
    if (lane == 0) bulk_wait_read_all();  // the previous image of this warp has been read
    __syncwarp();
    const uint32_t sel_lo = 0x3210u ^ (static_cast<uint32_t>(m7) * 0x1111u);
    const uint32_t sel_hi = 0x7654u ^ (static_cast<uint32_t>(m7) * 0x1111u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i0 = 2 * j, i1 = 2 * j + 1;
      const int l0 = h + 2 * (8 * ((i0 >> 2) & 1) + 4 * ((i0 >> 1) & 1) + 2 * (i0 & 1));
      const int l1 = h + 2 * (8 * ((i1 >> 2) & 1) + 4 * ((i1 >> 1) & 1) + 2 * (i1 & 1));
      const float ra = __shfl_sync(0xffffffffu, r, l0), rb = __shfl_sync(0xffffffffu, r, l1);
      if (path == kQuotMul) {
        const uint64_t nr2 = pk2(-ra, -rb);
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k][j] = mul2(x[k][j], nr2);
      } else {
        const float sa = __shfl_sync(0xffffffffu, s, l0), sb = __shfl_sync(0xffffffffu, s, l1);
        if (path == kQuotFma) {
          const uint64_t s2 = pk2(sa, sb), nr2 = pk2(-ra, -rb);
#pragma unroll
          for (int k = 0; k < 8; ++k) x[k][j] = quot2_fma(x[k][j], s2, nr2);
        } else {
          const TileDiv d0{sa, ra, make_tile_div_mode(sa)}, d1{sb, rb, make_tile_div_mode(sb)};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 f = unpk2(x[k][j]);
            x[k][j] = pk2(tile_quot(-f.x, d0), tile_quot(-f.y, d1));
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float q[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = e ? unpk2(x[k][j]).y : unpk2(x[k][j]).x;
        const uint32_t lo = e4m3x4_f(q[0], q[1], q[2], q[3]), hi = e4m3x4_f(q[4], q[5], q[6], q[7]);
        const uint32_t nlo = __byte_perm(lo, hi, sel_lo), nhi = __byte_perm(lo, hi, sel_hi);
        const int row = 8 * h + 2 * j + e;
        const uint32_t off = img + row * kTile + ((((m >> 1) ^ (row & 7)) << 4) | ((m & 1) << 3));
        *reinterpret_cast<uint2*>(quant_smem + off) = make_uint2(nlo, nhi);
      }
    }
    fence_async_shared();  // the image is read by a TMA store
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(sl.tmo, smem_u32(quant_smem) + img, tb * kTile, cb * kTile + 16 * wt, static_cast<int32_t>(g));
      bulk_commit();
    }
    return true;
  }

  static __device__ __forceinline__ void finish(const Args&, const Pipe&, int, int, State&) {}
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

// `tmo` is the output tensor map of ops that store through TMA (others
// ignore it).
template <class Op>
cudaError_t launch_pipe(const CUtensorMap& tm, const CUtensorMap& tmo, const typename Op::Args& a, const Pipe& p,
                        int num_sms, cudaStream_t stream) {
  static_assert(Layout<Op>::kSmem <= 227 * 1024, "shared memory budget");
  // 228 KB per SM, 1 KB of it reserved per CTA
  static_assert(Op::kCtasPerSm * (Layout<Op>::kSmem + 1024) <= 228 * 1024, "CTAs per SM");
  cudaError_t e = ensure_attr<Op>();
  if (e != cudaSuccess) return e;
  const int64_t ctas = static_cast<int64_t>(num_sms) * Op::kCtasPerSm;
  const int64_t grid = a.chunks < ctas ? a.chunks : ctas;
  e = launch_kernel(quant_pipe_kernel<Op>, dim3(static_cast<unsigned>(grid)), dim3(32 * (1 + Op::kWarps)),
                    Layout<Op>::kSmem, stream, tm, tmo, a, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

CUtensorMapDataType map_type(int esz) {
  return esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                  : (esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

constexpr int64_t kMaxBlocks = (1ll << 31) - 1;  // chunk indices are 32-bit in the walk

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
  if (chunks > kMaxBlocks) return cudaErrorInvalidValue;
  if (f32) {
    typename Quant1x128<true>::Args a{chunks, M, K, lds, KB, q, s, pow2};
    return launch_pipe<Quant1x128<true>>(tm, tm, a, p, l.num_sms, stream);
  }
  typename Quant1x128<false>::Args a{chunks, M, K, lds, KB, q, s, pow2};
  return launch_pipe<Quant1x128<false>>(tm, tm, a, p, l.num_sms, stream);
}

cudaError_t launch_quant_128x128(const void* w, bool f32, int64_t G, int64_t N, int64_t K, uint8_t* q, float* s,
                                 int pow2, const QuantLaunch& l, cudaStream_t stream) {
  const int esz = f32 ? 4 : 2;
  const int box_rows = f32 ? Quant128x128<true>::kBoxRows : Quant128x128<false>::kBoxRows;
  const int64_t NB = (N + kTile - 1) / kTile, KB = K / kTile;
  if (N > kMaxBlocks || KB > kMaxBlocks || G * NB * KB > kMaxBlocks) return cudaErrorInvalidValue;
  CUtensorMap tm;
  if (!make_map(&tm, map_type(esz), w, K, N, G, K * esz, N * K * esz, kTile, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const Pipe p{l.status, l.wait_limit_ns, l.debug_skip_fill};
  if (f32) {
    typename Quant128x128<true>::Args a{G * NB * KB, N, K, static_cast<int>(NB), static_cast<int>(KB), q, s, pow2};
    return launch_pipe<Quant128x128<true>>(tm, tm, a, p, l.num_sms, stream);
  }
  typename Quant128x128<false>::Args a{G * NB * KB, N, K, static_cast<int>(NB), static_cast<int>(KB), q, s, pow2};
  return launch_pipe<Quant128x128<false>>(tm, tm, a, p, l.num_sms, stream);
}

cudaError_t launch_requant_128x1(const void* src, int src_kind, const float* s_src, int64_t ld_t, int64_t G,
                                 int64_t T, int64_t C, const int32_t* valid_rows, uint8_t* qT, float* sT,
                                 int64_t ld_c, int pow2, const QuantLaunch& l, cudaStream_t stream) {
  const int esz = src_kind == 0 ? 1 : (src_kind == 1 ? 2 : 4);
  const int64_t TB = T / kTile, CB = C / kTile;
  if (TB * CB > kMaxBlocks || G * TB * CB > kMaxBlocks) return cudaErrorInvalidValue;
  // source as (32-byte column group, token, group, batch); one box is a tile
  const uint64_t cols = 32 / esz;
  const uint64_t dims[4] = {cols, static_cast<uint64_t>(T), static_cast<uint64_t>(C) / cols, static_cast<uint64_t>(G)};
  const uint64_t strides[3] = {static_cast<uint64_t>(C) * esz, 32, static_cast<uint64_t>(T * C) * esz};
  const uint32_t box[4] = {static_cast<uint32_t>(cols), kTile, static_cast<uint32_t>(kTile / cols), 1};
  CUtensorMap tm, tmo;
  if (!make_map4(&tm, map_type(esz), src, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  // qT [G][C][T]: one store box is a warp's 16 channel rows of 128 codes
  if (!make_map(&tmo, CU_TENSOR_MAP_DATA_TYPE_UINT8, qT, T, C, G, T, C * T, kTile, 16, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const Pipe p{l.status, l.wait_limit_ns, l.debug_skip_fill};
  const int tb = static_cast<int>(TB), cb = static_cast<int>(CB);
  switch (src_kind) {
    case 0: {
      typename Requant128x1<0>::Args a{G * TB * CB, T, C, ld_t, ld_c, tb, cb, s_src, valid_rows, sT, pow2};
      return launch_pipe<Requant128x1<0>>(tm, tmo, a, p, l.num_sms, stream);
    }
    case 1: {
      typename Requant128x1<1>::Args a{G * TB * CB, T, C, ld_t, ld_c, tb, cb, nullptr, valid_rows, sT, pow2};
      return launch_pipe<Requant128x1<1>>(tm, tmo, a, p, l.num_sms, stream);
    }
    default: {
      typename Requant128x1<2>::Args a{G * TB * CB, T, C, ld_t, ld_c, tb, cb, nullptr, valid_rows, sT, pow2};
      return launch_pipe<Requant128x1<2>>(tm, tmo, a, p, l.num_sms, stream);
    }
  }
}

}  // namespace fp8fg
