// FP8 GEMM with fine-grained scaling on fifth-generation tensor cores.
//
// What it computes (DeepSeek-V3 report excerpt, page 1, paragraph 3): FP8
// inputs, partial sums of each 128-wide K block promoted to FP32 registers
// on the CUDA cores and accumulated there in full FP32, output BF16 or FP32;
// operands carry 1x128 (activation) and 128x128 (weight) or 128x1 scales.
//
// How (sm_103a; the pages' Hopper design with two warpgroups ping-ponging
// WGMMA and promotion is replaced by):
//   warp 0      TMA producer: A tile 128x128, B tile BNx128 (both K-major,
//               128-byte swizzle), the 128 row scales of A and, for per-row
//               B scales, BN column scales, into an S-stage shared-memory
//               ring guarded by full/empty mbarriers;
//   warps 1, 2  MMA issuers, alternate K blocks: 4 x
//               tcgen05.mma.kind::f8f6f4 (K=32 each) per 128-K block into
//               one of several TMEM accumulator buffers, fresh per K block
//               (no accumulation across blocks), then a commit to the
//               buffer's "full" barrier (two issuers, because each MMA
//               costs its issuing thread a fixed time);
//   the rest    promotion + epilogue: tcgen05.ld the K block's FP32 partial
//               sums, acc += (sA[m,kb] * sB[n,kb]) * partial in registers,
//               release the TMEM buffer and the stage (whose scales they
//               read); after the last K block convert and store the tile
//               (BF16 or FP32, optional C += for FP32).
// Thread <-> data: each epilogue thread owns one row of the tile (its TMEM
// lane) and a contiguous group of columns, so the A scale is one scalar per
// thread per K block and the B block scale one scalar per warp.
// The kernel is persistent: one CTA per SM walks output tiles with stride
// gridDim.x, in M-fastest order so that concurrently running CTAs share the
// same B tiles in L2. Several TMEM buffers let the tensor core run ahead of
// the promotion warps; the shared-memory ring lets TMA run S blocks ahead.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "gemm_common.cuh"
#include "quant_math.cuh"
#include "kernels.h"
#include "launch.h"
#include "tmap.h"

namespace fp8fg {

namespace {

using namespace gemm_detail;

constexpr int kContigBand = 16;  // M blocks per raster band of the grouped-contiguous layout

// Tile configurations. The epilogue warps split the tile's columns in
// groups of kColsPerWarp; four warps (one per TMEM lane quarter) share a
// group. Register budget per thread is 65536 / (4 * ceil(warps / 4) * 32).
template <int BN>
struct Cfg {
  static constexpr int kColsPerWarp = (BN == 256) ? 128 : 64;
  static constexpr int kEpiWarps = 4 * BN / kColsPerWarp;   // 128: 8, 192: 12, 256: 8
  // BN=256: 12 warps. Warpgroup 0 (producer, MMA issuer, two idle warps)
  // hands registers to the two promotion warpgroups with setmaxnreg: a
  // promotion thread holds 128 FP32 accumulators, and at the 168 registers
  // of an even split the Stream-K variant spilled in its K loop. The launch
  // must hold kThreads x kRegsLaunch registers, and 128 x kRegsLow +
  // 256 x kRegsHigh must not exceed that (checked on the host against the
  // compiled register count before the first launch).
  static constexpr bool kRegSplit = (BN == 256);
  // MMA issuers: each tcgen05.mma costs its issuing thread a fixed ~50 ns
  // on top of the tensor core's work (measured: splitting a block's 4 MMAs
  // into 8 half-width ones adds ~23 ns per extra instruction), so with one
  // issuer a 128-wide block takes ~330 ns where the tensor core needs ~135.
  // A second issuer warp takes every other K block (its own TMEM buffer and
  // stage, its own commits). BN=256 uses warp 2, idle otherwise; BN=128 adds
  // a warp; BN=192 keeps one.
  static constexpr int kMaxIssuers = (BN == 192) ? 1 : 2;
  static constexpr int kEpiWarp0 = kRegSplit ? 4 : (BN == 128 ? 3 : 2);  // first promotion warp
  static constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
  static constexpr int kRegsLaunch = 168, kRegsLow = 48, kRegsHigh = 224;
  static_assert(!kRegSplit || (kEpiWarps == 8 && 128 * kRegsLow + 256 * kRegsHigh <= kThreads * kRegsLaunch),
                "register split exceeds the launch allocation");
  static constexpr int kAccBufs = (BN == 128) ? 4 : 2;      // TMEM partial-sum buffers
  static constexpr int kTmemCols = 512;                      // whole TMEM: one CTA per SM
  // BN=256 writes BF16 tiles through shared-memory staging and TMA stores:
  // each epilogue warp's 32 rows x 128 columns as two 128B-swizzled
  // 64-column boxes (8 KB). The first kBorrowWarps warps stage into the A
  // and B buffers of the tile's last pipeline stage, whose MMAs have
  // completed; that stage is released only once their stores have read it.
  // The other warps use a dedicated area. So the ring keeps all its stages.
  static constexpr bool kTmaStore = (BN == 256);
  static constexpr int kEpiWarpBytes = 32 * kColsPerWarp * 2;
  static constexpr int kBorrowWarps = kTmaStore ? (BM * BK + BN * BK) / kEpiWarpBytes : 0;  // 6
  static constexpr int kEpiBytes = kTmaStore ? (kEpiWarps - kBorrowWarps) * kEpiWarpBytes : 0;
  static constexpr int kStages = (BN == 128) ? 6 : (BN == 192 ? 5 : 4);
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = BN * BK;
  static constexpr int kSABytes = BM * 4;
  // B's scales of the stage's K block: one per column with row scales.
  // 128x128 block scales reach the promotion warps in one of two ways.
  // BN=192 and 256 (throughput-bound tiles): the producer copies the K
  // block's scale of each 128-column block the tile spans into the stage,
  // so a tile's first K block has nothing to fetch (a 192-wide tile may
  // start mid-block: two blocks either way). BN=128 (the decode-shaped,
  // latency-bound K loop, where any addition to a stage's refill showed
  // up in the time): each promotion warp loads its column block's scales
  // 128 K blocks at a time into its own staging area.
  static constexpr int kSBBytes = BN * 4;
  static constexpr bool kProducerScales = (BN != 128);
  static constexpr int kSbSpan = 2;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffEpi = kOffB + kStages * kBBytes;     // 1024-aligned (see assert)
  static constexpr int kOffSA = kOffEpi + kEpiBytes;
  static constexpr int kOffSB = kOffSA + kStages * kSABytes;
  static constexpr int kOffSbw = kOffSB + kStages * kSBBytes;      // per-warp block-scale staging
  static constexpr int kSbwChunk = 128;                            // K blocks staged at a time
  static constexpr int kOffBar = kOffSbw + (kProducerScales ? 0 : kEpiWarps * kSbwChunk * 4);
  // full[S], empty[S], tmem_full[B], tmem_empty[B], drain
  static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 1;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffTmemSlot + 16 + 1024;  // + alignment slack
  static_assert(kAccBufs * BN <= kTmemCols, "TMEM buffers exceed 512 columns");
  static_assert(kSmem > 116 * 1024, "keep one CTA per SM so the TMEM allocation never waits");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert((kOffB % 1024) == 0 && (kABytes % 1024) == 0 && (kBBytes % 1024) == 0,
                "128-byte swizzled tiles need 1024-byte alignment");
  static_assert(!kTmaStore || (kOffEpi % 1024) == 0, "swizzled store boxes need 1024-byte alignment");
};

template <int BN>
__device__ __forceinline__ Tile decode_tile(const KArgs& a, int t) {
  Tile ti;
  ti.tile = t;
  ti.sk_start = -1;
  // Uniform shortcuts for what dense problems (one group) and decode
  // shapes (one row block) would otherwise divide out: each division is a
  // dependent instruction sequence ahead of the producer's first copy.
  const int per_group = a.tiles_m * a.tiles_n;
  const int g = a.mode == kModeDense ? 0 : t / per_group;
  const int r = t - g * per_group;
  int mb, nb;
  if (a.mode == kModeContig) {
    // grouped raster: bands of kContigBand M blocks, M fastest inside a band.
    // A band's rows (a few experts) stay in L2 while its N blocks pass, and
    // each expert's B tiles are read about once per band. (M fastest over
    // all rows, as for dense problems, re-read the whole of A every wave.)
    const int band = r / (kContigBand * a.tiles_n);
    const int m_first = band * kContigBand;
    const int rows = a.tiles_m - m_first < kContigBand ? a.tiles_m - m_first : kContigBand;
    const int rr = r - band * kContigBand * a.tiles_n;
    mb = m_first + rr % rows;
    nb = rr / rows;
  } else if (a.tiles_m == 1) {
    mb = 0;
    nb = r;
  } else {
    mb = r % a.tiles_m;
    nb = r / a.tiles_m;
  }
  ti.m0 = mb * BM;
  ti.n0 = nb * BN;
  ti.kb0 = 0;
  ti.kbc = a.KB;
  ti.skip = false;
  ti.gA = ti.gB = ti.gC = 0;
  if (a.mode == kModeContig) {
    const int e = __ldg(a.m_indices + ti.m0);
    ti.gB = e;
    ti.skip = (e < 0) || (e >= a.groupsB);
  } else if (a.mode == kModeMaskedRows) {
    ti.gA = ti.gB = ti.gC = g;
    ti.skip = ti.m0 >= __ldg(a.masked + g);
  } else if (a.mode == kModeMaskedK) {
    ti.gA = ti.gB = ti.gC = g;
    int mk = __ldg(a.masked + g);
    mk = mk < 0 ? 0 : mk;
    const int kbc = (mk + BK - 1) / BK;
    ti.kbc = kbc < ti.kbc ? kbc : ti.kbc;
  }
  return ti;
}

// Masked rows: the active M blocks of group g, its first
// ceil(masked[g] / BM) (at most tiles_m).
__device__ __forceinline__ int masked_mblocks(const KArgs& a, int g) {
  int mk = __ldg(a.masked + g);
  mk = mk < 0 ? 0 : mk;
  const int mb = (mk + BM - 1) / BM;
  return mb < a.tiles_m ? mb : a.tiles_m;
}

// Masked rows: active tile j in group order, M blocks fastest inside a
// group, so that a group's M blocks read each B tile at about the same time.
// False when there are at most j active tiles.
template <int BN>
__device__ __forceinline__ bool decode_masked_tile(const KArgs& a, int j, Tile& ti) {
  const int groups = a.num_tiles / (a.tiles_m * a.tiles_n);
  for (int g = 0; g < groups; ++g) {
    const int mbs = masked_mblocks(a, g);
    if (j < mbs * a.tiles_n) {
      const int nb = j / mbs;
      ti = decode_tile<BN>(a, (g * a.tiles_n + nb) * a.tiles_m + (j - nb * mbs));
      return true;
    }
    j -= mbs * a.tiles_n;
  }
  return false;
}

// This CTA's work in order: whole tiles t = blockIdx.x + i * gridDim.x below
// dp_tiles (all tiles without Stream-K; for masked rows, the active tiles
// only, found from the device-side row counts, so that every CTA gets an
// equal share of real work), then its Stream-K unit range cut at tile
// boundaries into segments.
struct Work {
  int t, u, end;
};

// How a launch splits K: not at all (whole tiles), Stream-K (unit ranges
// cut at tile boundaries, partials summed through the workspace), or over
// the CTAs of a cluster (one tile per cluster, partials summed through
// distributed shared memory).
enum : int { kSplitNone = 0, kSplitStream = 1, kSplitCluster = 2 };

template <int kSK>
__device__ __forceinline__ Work work_begin(const KArgs& a) {
  Work w;
  w.t = blockIdx.x;
  w.u = w.end = 0;

  if constexpr (kSK == kSplitStream) {
    const int64_t u = static_cast<int64_t>(blockIdx.x) * a.sk_per_cta;
    const int64_t e = u + a.sk_per_cta;
    w.u = static_cast<int>(u < a.sk_units ? u : a.sk_units);
    w.end = static_cast<int>(e < a.sk_units ? e : a.sk_units);
  } else if constexpr (kSK == kSplitCluster) {
    // cluster t computes tile t; its CTA r (blockIdx.x % cl_split, the
    // rank: the clusters tile the grid along x) takes the r-th K range.
    // 32-bit unsigned arithmetic (the host splits only K < 2^24 blocks, so
    // (r + 1) * KB stays below 2^27): a 64-bit division is a long software
    // sequence ahead of the producer's first copy.
    const unsigned S = static_cast<unsigned>(a.cl_split), kb = static_cast<unsigned>(a.KB);
    const unsigned r = blockIdx.x % S;
    w.t = static_cast<int>(blockIdx.x / S);
    w.u = static_cast<int>(r * kb / S);
    w.end = static_cast<int>((r + 1) * kb / S);
  }
  return w;
}

// kCompact (masked rows only): the tiles are the active ones.
template <int BN, int kSK, bool kCompact>
__device__ __forceinline__ bool work_next(const KArgs& a, Work& w, Tile& ti) {
  if constexpr (kSK == kSplitCluster) {
    if (w.u >= w.end) return false;
    ti = decode_tile<BN>(a, w.t);
    ti.kb0 = w.u;
    ti.kbc = w.end - w.u;
    w.u = w.end;
    return true;
  }
  const int dp = kSK == kSplitStream ? a.dp_tiles : a.num_tiles;
  if constexpr (kCompact) {
    if (!decode_masked_tile<BN>(a, w.t, ti)) return false;
    w.t += gridDim.x;
    return true;
  }
  if (w.t < dp) {
    ti = decode_tile<BN>(a, w.t);
    w.t += gridDim.x;
    return true;
  }
  if constexpr (kSK == kSplitStream) {
    if (w.u < w.end) {
      const int tt = w.u / a.KB;
      const int kb0 = w.u - tt * a.KB;
      const int left = w.end - w.u;
      ti = decode_tile<BN>(a, a.sk_tile0 + tt);
      ti.kb0 = kb0;
      ti.kbc = left < a.KB - kb0 ? left : a.KB - kb0;
      ti.sk_start = w.u;
      w.u += ti.kbc;
      return true;
    }
  }
  return false;
}

// Stream-K slots: segments are numbered in unit order; a segment starting
// at unit s is preceded by the tile boundaries (multiples of KB) and CTA
// boundaries (multiples of sk_per_cta) in (0, s], counted by inclusion-
// exclusion over their common multiples (sk_lcm). A slot holds a BM x BN
// FP32 partial tile in the threads' register order, [warp][j/4][lane]
// float4, so every store and load of a warp is one contiguous 512-byte
// access.
__device__ __forceinline__ int64_t sk_slot(const KArgs& a, int s) {
  return static_cast<int64_t>(s / a.KB + s / a.sk_per_cta - s / a.sk_lcm);
}

// Store this segment's partials, count the arrival of this (tile, epilogue
// warp) and, in the warp that arrives last, replace acc by the sum of all
// pieces' partials in piece order (deterministic). Returns true in the warp
// that must store the final result. The counter is reset to 0 by that warp,
// so the workspace stays zeroed between calls.
template <int NC, int EW>
__device__ __forceinline__ bool sk_reduce(const KArgs& a, const Tile& ti, int row_in_tile, int ew, int lane,
                                          float (&acc)[NC]) {
  constexpr int64_t kSlot = static_cast<int64_t>(EW) * (NC / 4) * 32;  // float4 per slot
  const bool row_ok = ti.m0 + row_in_tile < a.rows;
  float4* ws4 = reinterpret_cast<float4*>(a.ws_partial) + static_cast<int64_t>(ew) * (NC / 4) * 32 + lane;
  if (row_ok) {
    float4* mine = ws4 + sk_slot(a, ti.sk_start) * kSlot;
#pragma unroll
    for (int j = 0; j < NC; j += 4) __stcg(mine + (j / 4) * 32, make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]));
  }
  __threadfence();
  __syncwarp();
  const int tt = ti.tile - a.sk_tile0;  // Stream-K tile index
  const int f = tt * a.KB;              // its first unit
  const int cf = f / a.sk_per_cta, cl = (f + a.KB - 1) / a.sk_per_cta;
  int* counter = a.ws_count + tt * 16 + ew;
  int prev = 0;
  if (lane == 0) prev = atomicAdd(counter, 1);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev != cl - cf) return false;
  __threadfence();
  if (lane == 0) *counter = 0;
#pragma unroll
  for (int j = 0; j < NC; ++j) acc[j] = 0.0f;
  if (row_ok) {
    for (int c = cf; c <= cl; ++c) {
      const float4* src = ws4 + sk_slot(a, c == cf ? f : c * a.sk_per_cta) * kSlot;
#pragma unroll
      for (int j = 0; j < NC; j += 4) {
        const float4 v = __ldcg(src + (j / 4) * 32);
        acc[j] += v.x; acc[j + 1] += v.y; acc[j + 2] += v.z; acc[j + 3] += v.w;
      }
    }
  }
  return true;
}

// Cluster split. The tile's 16 column chunks of 8 are divided among the S
// CTAs of its cluster, CTA r owning chunks [first(r), first(r + 1)),
// first(r) = floor(16 r / S). Each epilogue warp first writes its 32 rows
// x NC columns of FP32 partial sums into its own transpose area in this
// CTA's shared memory (the pipeline stages are idle once its K loop is
// done). Once every CTA of the cluster is past its K loop (a cluster
// barrier: from then on no stage of any of them is in use), the warp reads
// them back so that its lanes cover consecutive 16-byte pieces of an
// owner's rows, and stores them with st.shared::cluster into slot `rank` of
// the owner's receive area: one warp-wide store moves up to 512 contiguous
// bytes, where storing each lane's own row would scatter 32 pieces. After a
// second barrier (release and acquire: the stores have landed) every CTA
// sums its chunks over the S slots in rank order, so the result does not
// depend on timing, and stores them. Nothing reads another CTA's shared
// memory after that barrier, so a CTA may then leave.
// A transpose row is NC floats plus 16 bytes (an odd number of 16-byte
// units, so that the lanes' rows fall on distinct bank groups); a receive
// row is the widest share, ceil(16 / S) chunks.
constexpr int kMaxClusterSplit = 8;  // portable cluster size

template <int BN, int NC, int kEpiWarps>
struct ClusterPart {
  static constexpr int kChunks = BN / 8;
  static constexpr int kChunkBytes = 32;
  static constexpr int kMaxSplit = kMaxClusterSplit;
  static constexpr int kXposePitch = NC * 4 + 16;
  static constexpr int kXposeBytes = kEpiWarps * 32 * kXposePitch;
  static constexpr int kRecvOff = (kXposeBytes + 1023) / 1024 * 1024;
  static __host__ __device__ constexpr int recv_pitch(int S) { return (kChunks + S - 1) / S * kChunkBytes; }
  static constexpr int max_recv_bytes(int S = 2) {
    return S > kMaxSplit ? 0
                         : (S * BM * recv_pitch(S) > max_recv_bytes(S + 1) ? S * BM * recv_pitch(S)
                                                                            : max_recv_bytes(S + 1));
  }
  static constexpr int kBytes = kRecvOff + max_recv_bytes();
  static __host__ __device__ constexpr int first(int r, int S) { return r * kChunks / S; }
  // the owner of chunk ch: the r with first(r) <= ch < first(r + 1)
  static __device__ __forceinline__ int owner(int ch, int S) { return (ch * S + S - 1) / kChunks; }
};

// One epilogue warp's partial sums (rows row_base .. row_base + 31 of the
// tile, one per lane, columns col0 .. col0 + NC) into its transpose area.
template <class P, int NC>
__device__ __forceinline__ void cluster_stage(uint8_t* xpose, int lane, const float (&acc)[NC]) {
  float4* d = reinterpret_cast<float4*>(xpose + lane * P::kXposePitch);
#pragma unroll
  for (int j = 0; j < NC / 4; ++j) d[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
}

// The warp's staged rows, owner by owner, into the owners' receive areas.
template <class P, int NC>
__device__ __forceinline__ void cluster_push(const KArgs& a, const Tile& ti, int row_base, int col0, int lane,
                                             const uint8_t* xpose, uint32_t sbase) {
  const int S = a.cl_split;
  const int me = static_cast<int>(cluster_ctarank());
  const int valid = a.rows - (ti.m0 + row_base) < 32 ? a.rows - (ti.m0 + row_base) : 32;
  const int c0 = col0 / 8;
  const int pitch = P::recv_pitch(S);
  for (int r = P::owner(c0, S); r <= P::owner(c0 + NC / 8 - 1, S); ++r) {
    const int k_lo = c0 > P::first(r, S) ? c0 : P::first(r, S);
    const int k_hi = c0 + NC / 8 < P::first(r + 1, S) ? c0 + NC / 8 : P::first(r + 1, S);
    const int per_row = 2 * (k_hi - k_lo);  // 16-byte pieces of one row for this owner
    // p / per_row by multiplication (exact for p * per_row < 2^16)
    const uint32_t inv = (65536u + static_cast<uint32_t>(per_row) - 1) / static_cast<uint32_t>(per_row);
    const uint32_t dst = map_to_cta(sbase + P::kRecvOff, static_cast<uint32_t>(r)) +
                         static_cast<uint32_t>((me * BM + row_base) * pitch + (k_lo - P::first(r, S)) * P::kChunkBytes);
    const uint8_t* src = xpose + (k_lo - c0) * P::kChunkBytes;
    for (int p = lane; p < valid * per_row; p += 32) {
      const int row = static_cast<int>((static_cast<uint32_t>(p) * inv) >> 16);
      const int pc = p - row * per_row;
      const float4 v = *reinterpret_cast<const float4*>(src + row * P::kXposePitch + pc * 16);
      st_cluster_f4(dst + static_cast<uint32_t>(row * pitch + pc * 16), v.x, v.y, v.z, v.w);
    }
  }
}

// This CTA's chunks of the tile: the sum over the S slots of its receive
// area, stored to C.
template <class P, bool kF32>
__device__ __forceinline__ void cluster_reduce_store(const KArgs& a, const Tile& ti, const uint8_t* recv) {
  const int S = a.cl_split;
  const int r = static_cast<int>(cluster_ctarank());
  const int c_begin = P::first(r, S), nch = P::first(r + 1, S) - c_begin;
  const int pitch = P::recv_pitch(S);
  const int rows = a.rows - ti.m0 < BM ? a.rows - ti.m0 : BM;
  for (int i = threadIdx.x; i < rows * nch; i += blockDim.x) {
    const int row = i / nch;
    const int lc = i - row * nch;
    const int col = ti.n0 + (c_begin + lc) * 8;
    if (col >= a.N) continue;  // N % 8 == 0: a chunk is wholly inside or outside
    const uint8_t* src = recv + row * pitch + lc * P::kChunkBytes;
    float4 lo = make_float4(0.0f, 0.0f, 0.0f, 0.0f), hi = lo;
    for (int q = 0; q < S; ++q) {
      const float4 x = *reinterpret_cast<const float4*>(src + q * BM * pitch);
      const float4 y = *reinterpret_cast<const float4*>(src + q * BM * pitch + 16);
      lo.x += x.x; lo.y += x.y; lo.z += x.z; lo.w += x.w;
      hi.x += y.x; hi.y += y.y; hi.z += y.z; hi.w += y.w;
    }
    const int64_t o = static_cast<int64_t>(ti.m0 + row) * a.ldc + col;
    if constexpr (kF32) {
      float4* c = reinterpret_cast<float4*>(static_cast<float*>(a.C) + o);
      if (a.accumulate) {
        const float4 u = c[0], v = c[1];
        lo.x += u.x; lo.y += u.y; lo.z += u.z; lo.w += u.w;
        hi.x += v.x; hi.y += v.y; hi.z += v.z; hi.w += v.w;
      }
      c[0] = lo;
      c[1] = hi;
    } else {
      uint4 v;
      v.x = pack_bf16x2(lo.x, lo.y);
      v.y = pack_bf16x2(lo.z, lo.w);
      v.z = pack_bf16x2(hi.x, hi.y);
      v.w = pack_bf16x2(hi.z, hi.w);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.C) + o) = v;
    }
  }
}

// Fused 1x128 quantization of one epilogue warp's 32 rows x 128 columns of
// C (DeepSeek-V3 report excerpt, page 1, paragraph 3: activations are
// quantized per 1x128 tile; the DeepGEMM article's call to fuse the FP8 cast
// into the data movement, page 2, last paragraph). Every thread owns one
// row's 128 columns, one whole tile: the value quantized is C rounded to
// BF16 (what the unfused path writes and fp8_quant_1x128 then reads), the
// scale fl32(amax / 448) (or its power of two), the code E4M3(RN(x / s)) by
// the quantizer's own arithmetic, so the result is bit-identical to
// fp8_gemm_dense followed by fp8_quant_1x128. Codes go out through the
// warp's staging area (eight 16-byte chunks a row, 128-byte swizzle) and one
// TMA store; scales are stored directly, 32 consecutive floats a warp.
__device__ __forceinline__ void quant_store_tile(const KArgs& a, const Tile& ti, int row_in_tile, int col0, int lane,
                                                 uint8_t* region, const CUtensorMap* tmQ, float (&acc)[128]) {
  // BF16 rounding, packed in place (acc[i] <- the pair of columns 2i, 2i+1)
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const uint32_t w = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
    am = fmaxf(am, fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xFFFF0000u))));
    acc[i] = __uint_as_float(w);
  }
  const float s = tile_scale(am, a.pow2_out != 0);
  const float r = __frcp_rn(s);
  const int path = warp_quot_mode(make_tile_div_mode(s));
  // the staging area is free once earlier stores from it have read it
  if (lane == 0) bulk_wait_read_all();
  fence_async_shared();
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint64_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = neg_bf16x2(__float_as_uint(acc[c * 8 + i]));
    quot2_n<8>(v, path, s, r);
    uint4 o;
    o.x = e4m3x4_pk(v[0], v[1]);
    o.y = e4m3x4_pk(v[2], v[3]);
    o.z = e4m3x4_pk(v[4], v[5]);
    o.w = e4m3x4_pk(v[6], v[7]);
    *reinterpret_cast<uint4*>(region + lane * 128 + ((c ^ (lane & 7)) << 4)) = o;
  }
  fence_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_3d(tmQ, smem_u32(region), ti.n0 + col0, ti.m0 + (row_in_tile & ~31), 0);
    bulk_commit();
  }
  // a warp whose 128 columns lie wholly past N (the last tile of an N that
  // is not a multiple of 256) has no scale row to write
  const int row = ti.m0 + row_in_tile;
  if (row < a.rows && ti.n0 + col0 < a.N) a.s_out[static_cast<int64_t>((ti.n0 + col0) / 128) * a.ld_s + row] = s;
}

// Kernel variants besides the plain one: fused 1x128 quantization of the
// output, or B read MN-major (the weight as its own transpose).
enum : int { kVarPlain = 0, kVarQuant = 1, kVarBT = 2 };

template <int BN, bool kBRow, bool kF32, int kSplit, bool kCompact, int kVar>
__global__ void __launch_bounds__(Cfg<BN>::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmQ,
                    const KArgs a) {
  constexpr bool kQ = kVar == kVarQuant;
  constexpr bool kBT = kVar == kVarBT;
  static_assert(!kQ || (BN == 256 && !kBRow && !kF32 && !kCompact),
                "fused quantization: 128-column warps of BF16 output, dense layout");
  static_assert(!kBT || (BN != 192 && !kBRow && !kCompact), "MN-major B: 128-column boxes, block scales");
  static_assert(kSplit != kSplitCluster || (BN == 128 && !kQ && !kCompact),
                "cluster split: 128-column tiles, row-by-row stores, dense layout");
  using C = Cfg<BN>;
  using CP = ClusterPart<BN, C::kColsPerWarp, C::kEpiWarps>;
  static_assert(kSplit != kSplitCluster || CP::kBytes <= C::kOffEpi,
                "the transpose and receive areas fit in the pipeline stages");
  constexpr int S = C::kStages;
  constexpr int NB = C::kAccBufs;
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
  auto tfull_bar = [bar0](uint32_t b) { return bar0 + (2 * S + b) * 8; };
  auto tempty_bar = [bar0](uint32_t b) { return bar0 + (2 * S + NB + b) * 8; };
  const uint32_t drain_bar = bar0 + (2 * S + 2 * NB) * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSA);
    if (kBRow) prefetch_tmap(&tmSB);
    for (int s = 0; s < S; ++s) {
      // the producer's expect-tx arrival, and with block scales of B the
      // arrival of its copies of them (below)
      mbar_init(full_bar(s), (!kBRow && C::kProducerScales) ? 2 : 1);
      // a stage is free once every promotion warp has seen its K block's MMAs
      // complete (tmem_full) and has read its scales: the MMA issuer does not
      // need to commit to it, which keeps its per-block loop short
      mbar_init(empty_bar(s), C::kEpiWarps);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), C::kEpiWarps);
    }
    mbar_init(drain_bar, static_cast<uint32_t>(a.mma_issuers));
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  grid_dependency_sync();

  if (warp < C::kEpiWarp0) {
   if constexpr (C::kRegSplit) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsLow));
   if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t tx = static_cast<uint32_t>(a.a_rows_box) * BK + C::kBBytes + C::kSABytes + (kBRow ? C::kSBBytes : 0);
      uint32_t it = 0;
      bool ok = true;
      Work wk = work_begin<kSplit>(a);
      Tile ti;
      while (ok && work_next<BN, kSplit, kCompact>(a, wk, ti)) {
        if (ti.skip) continue;
        // B's block scales of the tile's first 128-column block (BN=192
        // and 256: the tile spans two)
        const int nb0 = ti.n0 / 128;
        const float* sbt = a.sB + static_cast<int64_t>(ti.gB) * a.sb_nblk * a.sb_kblk +
                           static_cast<int64_t>(nb0) * a.sb_col_stride;
        for (int kb = ti.kb0; kb < ti.kb0 + ti.kbc; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1;
          if (!mbar_wait(empty_bar(s), ph ^ 1, a.status, kStatusTimeoutProducer, a.wait_limit_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), tx);
          if (static_cast<int>(it) == a.debug_skip_fill) continue;  // test hook: never filled
          tma_load_3d(sbase + C::kOffA + s * C::kABytes, &tmA, full_bar(s), kb * BK, ti.m0, ti.gA);
          if constexpr (kBT) {
            // [K][N] rows: boxes of 128 columns x 128 K, one per 128 columns
#pragma unroll
            for (int j = 0; j < BN / 128; ++j)
              tma_load_3d(sbase + C::kOffB + s * C::kBBytes + j * 128 * BK, &tmB, full_bar(s), ti.n0 + j * 128,
                          kb * BK, ti.gB);
          } else {
            tma_load_3d(sbase + C::kOffB + s * C::kBBytes, &tmB, full_bar(s), kb * BK, ti.n0, ti.gB);
          }
          tma_load_3d(sbase + C::kOffSA + s * C::kSABytes, &tmSA, full_bar(s), ti.m0, kb, ti.gA);
          if (kBRow)
            tma_load_3d(sbase + C::kOffSB + s * C::kSBBytes, &tmSB, full_bar(s), ti.n0, kb, ti.gB);
          if constexpr (!kBRow && C::kProducerScales) {
            // B's 128x128 block scales of this K block, one per 128-column
            // block of the tile, copied into the stage beside A's scales
            // (zero for a block past N): the promotion warps read them
            // there, with nothing to fetch at a tile's first K block
            const float* sbk = sbt + static_cast<int64_t>(kb) * a.sb_red_stride;
#pragma unroll
            for (int j = 0; j < C::kSbSpan; ++j) {
              const bool in = nb0 + j < a.sb_nblk;
              cp_async_4(sbase + C::kOffSB + s * C::kSBBytes + j * 4, in ? sbk + j * a.sb_col_stride : a.sB,
                         in ? 4u : 0u);
            }
            cp_async_mbar_arrive_noinc(full_bar(s));
          }
        }
      }
      // No copy may still be landing in shared memory when the CTA exits:
      // wait (bounded, ignoring the error word) for the last fill of each stage.
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
      for (uint32_t i = first; i < it; ++i) {
        mbar_wait(full_bar(i % S), (i / S) & 1, nullptr, 0, a.wait_limit_ns);
      }
      cp_async_wait_all();
    }
   } else if (warp == 1 || (C::kMaxIssuers > 1 && warp == 2)) {
    // ------------------------------------------------------------ MMA issuers
    // issuer i of a.mma_issuers (1 or 2) takes the K blocks it with
    // it % a.mma_issuers == i
    const uint32_t issuer = static_cast<uint32_t>(warp - 1);
    const uint32_t nis = static_cast<uint32_t>(a.mma_issuers);
    if (lane == 0 && issuer < nis) {
      constexpr uint32_t idesc = f8_idesc(BM, BN, kBT);
      uint32_t it = 0;
      bool ok = true;
      Work wk = work_begin<kSplit>(a);
      Tile ti;
      while (ok && work_next<BN, kSplit, kCompact>(a, wk, ti)) {
        if (ti.skip) continue;
        for (int kb = ti.kb0; kb < ti.kb0 + ti.kbc; ++kb, ++it) {
          if ((it & (nis - 1)) != issuer) continue;  // the other issuer's block
          const uint32_t s = it % S, ph = (it / S) & 1;
          const uint32_t buf = it % NB, tph = (it / NB) & 1;
          if (!mbar_wait(tempty_bar(buf), tph ^ 1, a.status, kStatusTimeoutMma, a.wait_limit_ns) ||
              !mbar_wait(full_bar(s), ph, a.status, kStatusTimeoutMma, a.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = kmajor_sw128_desc(sbase + C::kOffA + s * C::kABytes);
          // K-major B advances 32 bytes along its rows per MMA; MN-major B
          // 32 rows of 128 bytes (descriptor units of 16 bytes)
          const uint64_t bd = kBT ? mnmajor_sw128_desc(sbase + C::kOffB + s * C::kBBytes, 128 * BK)
                                  : kmajor_sw128_desc(sbase + C::kOffB + s * C::kBBytes);
          constexpr uint64_t kBStep = kBT ? (32 * 128) >> 4 : 32 >> 4;
          const uint32_t d = tmem_base + buf * BN;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            // advance 32 bytes (= 32 E4M3 elements) along K inside the swizzle atom
            mma_f8f6f4(d, ad + 2 * k, bd + kBStep * k, idesc, k > 0 ? 1u : 0u);
          }
          mma_commit(tfull_bar(buf));
        }
      }
      // All MMAs issued by the issuers complete before TMEM is released
      // (the drain barrier counts one commit per issuer).
      mma_commit(drain_bar);
      if (!mbar_wait(drain_bar, 0, nullptr, 0, a.wait_limit_ns)) atomicCAS(a.status, 0u, kStatusTimeoutDrain);
    }
   }
  } else {
    if constexpr (C::kRegSplit) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsHigh));
    // ------------------------------------------------------------ promotion + epilogue
    constexpr int NC = C::kColsPerWarp;
    const int ew = warp - C::kEpiWarp0;
    const int quarter = warp & 3;               // TMEM lanes this warp may access
    const int col0 = (ew >> 2) * NC;            // column group of the tile
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const float* smem_sa = reinterpret_cast<const float*>(smem + C::kOffSA);
    const float* smem_sb = reinterpret_cast<const float*>(smem + C::kOffSB);
    // BN=128: block scales of this warp's column group, staged 128 K blocks
    // at a time by the warp itself (no cross-warp barrier that a warp
    // leaving on the error path could leave waiting)
    float* sbw = reinterpret_cast<float*>(smem + C::kOffSbw) + ew * C::kSbwChunk;
    float acc[NC];
    uint32_t it = 0;
    bool ok = true;
    bool pushed = false;  // cluster split: this warp has passed the first cluster barrier
    // BF16 tiles go out through shared-memory staging and TMA stores
    constexpr bool kStage = C::kTmaStore;
    int held = -1;  // pipeline stage kept for staging (kStage, warps < kBorrowWarps)
    // The previous tile's staging stage, released once this tile's first K
    // block is promoted: by then its stores have normally read it, so the
    // wait for that read no longer sits between the epilogue and the next
    // tile's first promotion (where every warp's buffer release gates the
    // MMA). The producer needs the stage again only S blocks later.
    int prev_held = -1;
    bool prev_staged = false;
    // (BF16 tiles of the dense and contiguous layouts, where it was
    // measured faster: 16-block tiles of K=2048 ~4%; FP32 C, whose two
    // staging rounds per tile already wait on the first round's read, the
    // masked-rows kernel and the fused quantization were slower with it)
    constexpr bool kDeferRelease = kStage && !kF32 && !kCompact && !kQ;
    Work wk = work_begin<kSplit>(a);
    Tile ti;
    while (ok && work_next<BN, kSplit, kCompact>(a, wk, ti)) {
      if (ti.skip) continue;
#pragma unroll
      for (int j = 0; j < NC; ++j) acc[j] = 0.0f;
      // this warp's 128-column block, counted from the tile's first (its
      // slot among the stage's block scales of B)
      const int sb_slot = (ti.n0 + col0) / 128 - ti.n0 / 128;
      // the tile's K blocks kb0 .. kb0+kbc-1 by their offset jb in its range:
      // written this way the loop compiles the same whether kb0 is the
      // constant 0 (whole tiles) or the start of a split's K range
      const int kb0 = ti.kb0, kbc = ti.kbc;
      for (unsigned jb = 0; jb < static_cast<unsigned>(kbc); ++jb, ++it) {
        const uint32_t s = it % S, ph = (it / S) & 1;
        const uint32_t buf = it % NB, tph = (it / NB) & 1;
        if (!kBRow && !C::kProducerScales && (jb % C::kSbwChunk) == 0) {
          const int nbk = (ti.n0 + col0) / 128;
          const float* src = a.sB + static_cast<int64_t>(ti.gB) * a.sb_nblk * a.sb_kblk +
                             static_cast<int64_t>(nbk) * a.sb_col_stride + static_cast<int64_t>(kb0) * a.sb_red_stride;
          __syncwarp();
#pragma unroll
          for (int i = 0; i < C::kSbwChunk / 32; ++i) {
            const unsigned k = jb + i * 32 + lane;
            sbw[i * 32 + lane] =
                (nbk < a.sb_nblk && k < static_cast<unsigned>(kbc)) ? __ldg(src + static_cast<int64_t>(k) * a.sb_red_stride)
                                                                    : 0.0f;
          }
          __syncwarp();
        }
        bool got = mbar_wait(tfull_bar(buf), tph, a.status, kStatusTimeoutEpilogue, a.wait_limit_ns);
        got = got && mbar_wait(full_bar(s), ph, a.status, kStatusTimeoutEpilogue, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const float sa = smem_sa[s * BM + row_in_tile];
        float sc = 0.0f;
        if constexpr (!kBRow) sc = sa * (C::kProducerScales ? smem_sb[s * BN + sb_slot] : sbw[jb % C::kSbwChunk]);
        const float* sbv = smem_sb + s * BN + col0;
        const uint32_t taddr = tmem_base + lane_bits + buf * BN + col0;
        tc_fence_after();
        if constexpr (NC == 64 && C::kThreads <= 320) {
          uint32_t r[64];
          tmem_ld64(taddr, r);
          promote<64, kBRow>(acc, r, sc, sa, sbv);
        } else if constexpr (NC == 64) {
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t r[32];
            tmem_ld32(taddr + ch * 32, r);
            promote<32, kBRow>(acc + ch * 32, r, sc, sa, sbv + ch * 32);
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < NC / 16; ++ch) {
            uint32_t r[16];
            tmem_ld16(taddr + ch * 16, r);
            promote<16, kBRow>(acc + ch * 16, r, sc, sa, sbv + ch * 16);
          }
        }
        tc_fence_before();
        __syncwarp();
        // the staging warps keep the tile's last stage for the epilogue
        const bool hold = kStage && ew < C::kBorrowWarps && jb + 1 == static_cast<unsigned>(kbc);
        if (hold) held = static_cast<int>(s);
        if (lane == 0) {
          if (!hold) mbar_arrive(empty_bar(s));
          mbar_arrive(tempty_bar(buf));
        }
        if constexpr (kDeferRelease) {
          if (prev_held >= 0) {
            if (lane == 0) {
              if (prev_staged) bulk_wait_read_all();
              mbar_arrive(empty_bar(prev_held));
            }
            prev_held = -1;
          }
        }
      }
      if (!ok) break;
      bool store = !(a.accumulate && ti.kbc == 0);
      if constexpr (kSplit == kSplitStream) {
        // a Stream-K piece of a split tile: only the last to arrive stores
        if (ti.kbc != a.KB) store = sk_reduce<NC, C::kEpiWarps>(a, ti, row_in_tile, ew, lane, acc);
      } else if constexpr (kSplit == kSplitCluster) {
        // this warp's partial into its transpose area (its own stages are
        // free: every MMA has completed and every fill has landed, the
        // fence orders the tensor core's reads of them before these
        // writes); then the first cluster barrier: every CTA of the cluster
        // is past its K loop, so the owners' receive areas are free too
        uint8_t* xpose = smem + ew * 32 * CP::kXposePitch;
        fence_async_shared();
        cluster_stage<CP, NC>(xpose, lane, acc);
        __syncwarp();
        cluster_sync();
        pushed = true;
        cluster_push<CP, NC>(a, ti, quarter * 32, col0, lane, xpose, sbase);
        store = false;
      }
      bool staged = false;
      if (store) {
        if constexpr (kStage) {
          // Staging area: the first kBorrowWarps warps borrow the stage they
          // kept from the tile's last K block; the others own a dedicated
          // area. A tile without K blocks (an expert with no tokens in the
          // masked-K layout) kept no stage: those warps store row by row.
          uint8_t* region = nullptr;
          if (held >= 0 && ew < 2)
            region = smem + C::kOffA + held * C::kABytes + ew * C::kEpiWarpBytes;
          else if (held >= 0)
            region = smem + C::kOffB + held * C::kBBytes + (ew - 2) * C::kEpiWarpBytes;
          else if (ew >= C::kBorrowWarps)
            region = smem + C::kOffEpi + (ew - C::kBorrowWarps) * C::kEpiWarpBytes;
          if constexpr (kQ) {
            // BF16 C (if asked for), then its 1x128 quantization through the
            // same staging area
            if (a.c_bf16) staged = store_tile_tma<NC, false>(a, ti, row_in_tile, col0, lane, region, &tmC, acc);
            quant_store_tile(a, ti, row_in_tile, col0, lane, region, &tmQ, acc);
            staged = true;
          } else {
            if (region != nullptr) staged = store_tile_tma<NC, kF32>(a, ti, row_in_tile, col0, lane, region, &tmC, acc);
          }
        }
        if (!staged) store_row<NC, kF32>(a, ti, row_in_tile, col0, acc);
      }
      if (held >= 0) {
        if constexpr (kDeferRelease) {
          // released after the next tile's first K block (above), or
          // below if there is none
          prev_held = held;
          prev_staged = staged;
        } else {
          // release the borrowed stage once this warp's stores have read it
          if (lane == 0) {
            if (staged) bulk_wait_read_all();
            mbar_arrive(empty_bar(held));
          }
        }
        held = -1;
      }
    }
    if (prev_held >= 0 && lane == 0) {
      if (prev_staged) bulk_wait_read_all();
      mbar_arrive(empty_bar(prev_held));
    }
    // no store may still be reading shared memory when the CTA exits
    if constexpr (kStage) {
      if (lane == 0) bulk_wait_all();
    }
    if constexpr (kSplit == kSplitCluster) {
      // a warp that left its loop early (a timed-out wait) still takes part
      // in the first barrier, so that no CTA of the cluster waits forever
      if (!pushed) {
        __syncwarp();
        fence_async_shared();
        cluster_sync();
      }
    }
  }

  if constexpr (kSplit == kSplitCluster) {
    // the producer and MMA warps take part in the first barrier here; then
    // every thread: the second barrier (all partials have landed), and this
    // CTA's share of the tile
    __syncwarp();
    if (warp < C::kEpiWarp0) {
      fence_async_shared();
      cluster_sync();
    }
    cluster_sync();
    cluster_reduce_store<CP, kF32>(a, decode_tile<BN>(a, static_cast<int>(blockIdx.x / a.cl_split)),
                                   smem + CP::kRecvOff);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

// Raise the kernel's dynamic shared-memory limit once per device (the call
// costs tens of microseconds of host time, so it is not repeated per launch).
template <int BN, bool kBRow, bool kF32, int kSplit, bool kCompact, int kVar = kVarPlain>
cudaError_t ensure_smem_attr() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  using C = Cfg<BN>;
  if constexpr (C::kRegSplit) {
    // setmaxnreg.inc waits until the block's launch allocation can cover the
    // raised counts, forever if it never can: refuse to launch a build whose
    // register count does not cover the split.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fp8_gemm_kernel<BN, kBRow, kF32, kSplit, kCompact, kVar>);
    if (e != cudaSuccess) return e;
    if (static_cast<long>(fa.numRegs) * C::kThreads < 128L * C::kRegsLow + 256L * C::kRegsHigh)
      return cudaErrorInvalidConfiguration;
  }
  e = cudaFuncSetAttribute(fp8_gemm_kernel<BN, kBRow, kF32, kSplit, kCompact, kVar>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<BN>::kSmem);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Work plan of a launch. Without Stream-K: one whole tile per work item,
// min(tiles, SMs) CTAs. Stream-K (dense only) for decode-sized problems
// (tiles <= SMs/2) when the caller's workspace holds the partials: every
// tile is split along K over up to all SMs, at least kMinUnits K blocks per
// CTA. (Splitting only the last, partly idle wave of larger problems was
// measured slower than leaving it: the split tiles' FP32 partial stores and
// the summing cost more than the idle SMs did.)
struct Plan {
  bool sk = false;
  int grid = 0;
  int dp_tiles = 0;
  int64_t sk_units = 0, sk_per_cta = 0, sk_lcm = 0;
  size_t partial_bytes = 0, count_bytes = 0;
};

constexpr int64_t kMinUnits = 4;

// Workspace layout: arrival counters first, in a region of fixed size (16
// per split tile, at most num_sms / 2 split tiles), then the partial tiles.
// The counter region only ever holds counters, which every call returns to
// zero, so calls whose plans differ (tile width, shape) can share one
// workspace: none of them finds another's partial sums where it counts.
size_t counter_region_bytes(int num_sms) {
  return (static_cast<size_t>(num_sms / 2) * 16 * sizeof(int) + 255) / 256 * 256;
}

int64_t gcd64(int64_t x, int64_t y) {
  while (y != 0) {
    const int64_t t = x % y;
    x = y;
    y = t;
  }
  return x;
}

Plan plan_gemm(int mode, int64_t rows, int64_t N, int64_t K, int64_t groups, int num_sms, int bn,
               size_t ws_avail) {
  Plan p;
  const int64_t KB = K / BK;
  const int64_t tiles = groups * ((rows + BM - 1) / BM) * ((N + bn - 1) / bn);
  p.grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  p.dp_tiles = static_cast<int>(tiles);
  if (mode != kModeDense || groups != 1 || tiles <= 0 || KB <= 0) return p;
  const int64_t dp = 0;
  if (tiles * 2 > num_sms) return p;
  const int64_t cap = tiles * KB / kMinUnits;
  const int64_t grid = cap < num_sms ? cap : num_sms;
  if (grid < 2 * tiles) return p;  // too little K to split usefully
  const int64_t units = (tiles - dp) * KB;
  if (units >= (1ll << 31)) return p;  // device-side unit counters are 32-bit
  const int64_t per = (units + grid - 1) / grid;
  const int64_t lcm = KB / gcd64(KB, per) * per;
  const int64_t segs = 1 + (units - 1) / KB + (units - 1) / per - (units - 1) / lcm;
  const size_t partial = static_cast<size_t>(segs) * BM * bn * sizeof(float);
  const size_t counts = counter_region_bytes(num_sms);
  if (static_cast<size_t>(tiles - dp) * 16 * sizeof(int) > counts || partial + counts > ws_avail) return p;
  p.sk = true;
  p.grid = static_cast<int>((units + per - 1) / per);
  p.dp_tiles = static_cast<int>(dp);
  p.sk_units = units;
  p.sk_per_cta = per;
  p.sk_lcm = lcm;
  p.partial_bytes = partial;
  p.count_bytes = counts;
  return p;
}

// Split policy for decode-sized dense problems: automatic (the cluster
// split wherever it applies, else Stream-K when a workspace is given),
// Stream-K only, or the cluster split whenever it applies. FP8FG_SPLIT=
// stream|cluster sets it at load; fp8fg_debug_set(4, ...) at run time.
enum : int { kPolicyAuto = 0, kPolicyStream = 1, kPolicyCluster = 2 };
std::atomic<int> g_split_policy{[] {
  const char* v = std::getenv("FP8FG_SPLIT");
  if (v && std::strcmp(v, "stream") == 0) return static_cast<int>(kPolicyStream);
  if (v && std::strcmp(v, "cluster") == 0) return static_cast<int>(kPolicyCluster);
  return static_cast<int>(kPolicyAuto);
}()};

int split_policy() { return g_split_policy.load(std::memory_order_relaxed); }

// Two MMA issuers where the tile configuration has room for them
// (FP8FG_ISSUERS=1 keeps one, for timing comparisons).
bool two_issuers_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("FP8FG_ISSUERS");
    return !(v && v[0] == '1');
  }();
  return on;
}

// Clusters of `size` CTAs of `fn` that fit on the device at once (cached per
// device and size; the kernels that share a tile configuration have the same
// threads and shared memory, so one query serves them all).
template <class Fn>
cudaError_t cluster_capacity(Fn fn, int size, int* fit) {
  static std::atomic<int> cache[64][kMaxClusterSplit + 1];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::atomic<int>& slot = cache[dev & 63][size];
  const int v = slot.load(std::memory_order_acquire);
  if (v > 0) {
    *fit = v - 1;
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(size));
  cfg.blockDim = dim3(Cfg<128>::kThreads);
  cfg.dynamicSmemBytes = Cfg<128>::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(size);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
  if (e != cudaSuccess) return e;
  slot.store(n + 1, std::memory_order_release);
  *fit = n;
  return cudaSuccess;
}

// Cluster split of a decode-sized dense problem (its 128 x 128 tiles at most
// half the SMs): the largest S <= 8 with S CTAs per tile on the SMs, at
// least kMinUnits K blocks per CTA, and all tiles' clusters resident at
// once. *cl = 0 where none applies.
template <class Fn>
cudaError_t pick_cluster_split(int mode, int64_t rows, int64_t N, int64_t K, int64_t groups, int num_sms, Fn fn,
                               int* cl) {
  *cl = 0;
  if (mode != kModeDense || groups != 1) return cudaSuccess;
  const int64_t KB = K / BK;
  if (KB >= (int64_t{1} << 24)) return cudaSuccess;  // the device splits K in 32 bits
  const int64_t tiles = ((rows + BM - 1) / BM) * ((N + 127) / 128);
  if (tiles <= 0 || tiles * 2 > num_sms) return cudaSuccess;
  int64_t S = num_sms / tiles;
  if (S > kMaxClusterSplit) S = kMaxClusterSplit;
  if (S > KB / kMinUnits) S = KB / kMinUnits;
  for (; S >= 2; --S) {
    int fit = 0;
    const cudaError_t e = cluster_capacity(fn, static_cast<int>(S), &fit);
    if (e != cudaSuccess) return e;
    if (fit >= tiles) break;
  }
  *cl = S >= 2 ? static_cast<int>(S) : 0;
  return cudaSuccess;
}

template <int BN>
bool encode_maps(const GemmProblem& p, MapSet* m) {
  using C = Cfg<BN>;
  const int64_t KB = p.K / BK;
  const int64_t groupsA = (p.mode == kModeMaskedRows || p.mode == kModeMaskedK) ? p.groups : 1;
  bool ok = make_map(&m->a, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.A, p.K, p.rows, groupsA, p.K, p.rows * p.K, BK,
                     a_box_rows(p.rows), CU_TENSOR_MAP_SWIZZLE_128B);
  if (p.b_mn_major)  // B stored [K][N]: boxes of 128 columns x 128 K rows
    ok = ok && make_map(&m->b, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.B, p.N, p.K, p.groupsB, p.N, p.N * p.K, 128, BK,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  else
    ok = ok && make_map(&m->b, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.B, p.K, p.N, p.groupsB, p.K, p.N * p.K, BK, BN,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&m->sa, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.sA, p.rows, KB, groupsA, ld4(p.rows) * 4,
                      KB * ld4(p.rows) * 4, BM, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (p.b_row) {
    ok = ok && make_map(&m->sb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.sB, p.N, KB, p.groupsB, ld4(p.N) * 4,
                        KB * ld4(p.N) * 4, BN, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    m->sb = m->sa;  // unused
  }
  const int64_t groupsC = groupsA;
  if (C::kTmaStore && p.C != nullptr) {
    const int64_t esz = p.out_f32 ? 4 : 2;
    ok = ok && make_map(&m->c, p.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.C,
                        p.N, p.rows, groupsC, p.N * esz, p.rows * p.N * esz, 128 / esz, 32,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    m->c = m->sa;  // unused
  }
  if (p.q_out != nullptr) {
    ok = ok && make_map(&m->q, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.q_out, p.N, p.rows, 1, p.N, p.rows * p.N, 128, 32,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    m->q = m->sa;  // unused
  }
  return ok;
}

template <int BN>
bool get_maps(const GemmProblem& p, MapSet* out) {
  MapKey k;
  std::memset(&k, 0, sizeof(k));  // padding bytes take part in the comparison
  const int64_t groupsA = (p.mode == kModeMaskedRows || p.mode == kModeMaskedK) ? p.groups : 1;
  k.A = p.A; k.B = p.B; k.sA = p.sA; k.sB = p.b_row ? p.sB : nullptr; k.C = p.C; k.Q = p.q_out;
  k.rows = p.rows; k.N = p.N; k.K = p.K; k.groupsA = groupsA; k.groupsB = p.groupsB; k.groupsC = groupsA;
  k.kind = p.b_mn_major ? -BN : BN; k.b_row = p.b_row; k.out_f32 = p.out_f32;
  if (map_cache_find(k, out)) return true;
  if (!encode_maps<BN>(p, out)) return false;
  map_cache_put(k, *out);
  return true;
}

template <int BN>
cudaError_t launch_bn(const GemmProblem& p, uint32_t* status, uint64_t wait_limit_ns, int debug_skip_fill,
                      int num_sms, cudaStream_t stream, const char** detail) {
  using C = Cfg<BN>;
  const int64_t KB = p.K / BK;
  MapSet ms;
  if (!get_maps<BN>(p, &ms)) {
    *detail = "cuTensorMapEncodeTiled failed (driver entry point missing or arguments rejected)";
    return cudaErrorInvalidValue;
  }
  const CUtensorMap& tmA = ms.a;
  const CUtensorMap& tmB = ms.b;
  const CUtensorMap& tmSA = ms.sa;
  const CUtensorMap& tmSB = ms.sb;
  const CUtensorMap& tmC = ms.c;
  const CUtensorMap& tmQ = ms.q;
  KArgs a;
  a.mode = p.mode;
  a.KB = static_cast<int>(KB);
  a.rows = static_cast<int>(p.rows);
  a.N = static_cast<int>(p.N);
  a.K = static_cast<int>(p.K);
  a.tiles_m = static_cast<int>((p.rows + BM - 1) / BM);
  a.tiles_n = static_cast<int>((p.N + BN - 1) / BN);
  const int64_t nt = p.groups * a.tiles_m * a.tiles_n;
  if (nt > 0x7FFFFFFF) {
    *detail = "too many output tiles";
    return cudaErrorInvalidValue;
  }
  a.num_tiles = static_cast<int>(nt);
  a.groupsB = static_cast<int>(p.groupsB);
  a.accumulate = p.accumulate;
  a.m_indices = p.m_indices;
  a.masked = p.masked;
  a.sB = p.sB;
  a.sb_nblk = static_cast<int>((p.N + 127) / 128);
  a.sb_kblk = static_cast<int>(KB);
  a.sb_col_stride = p.b_mn_major ? 1 : a.sb_kblk;
  a.sb_red_stride = p.b_mn_major ? a.sb_nblk : 1;
  a.C = p.C;
  a.ldc = p.N;
  a.c_group_stride = p.rows * p.N;
  a.status = status;
  a.wait_limit_ns = wait_limit_ns;
  a.debug_skip_fill = debug_skip_fill;
  a.dp_tiles = a.num_tiles;
  a.sk_tile0 = 0;
  a.sk_units = a.sk_per_cta = a.sk_lcm = 0;
  a.ws_partial = nullptr;
  a.ws_count = nullptr;
  a.cl_split = 0;
  a.mma_issuers = (C::kMaxIssuers > 1 && two_issuers_enabled()) ? 2 : 1;
  a.a_rows_box = a_box_rows(p.rows);
  a.s_out = p.s_out;
  a.ld_s = ld4(p.rows);
  a.pow2_out = p.pow2_out;
  a.c_bf16 = p.C != nullptr;
  if (a.num_tiles == 0) return cudaSuccess;
  const Plan plan = plan_gemm(p.mode, p.rows, p.N, p.K, p.groups, num_sms, BN,
                              p.workspace != nullptr ? p.workspace_bytes : 0);

  using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, KArgs);
  // whole tiles / Stream-K / active tiles of the masked-rows layout / cluster split
  KernelFn kernels[4] = {nullptr, nullptr, nullptr, nullptr};
  cudaError_t (*cluster_attr)() = nullptr;
  const bool masked = p.mode == kModeMaskedRows;
  cudaError_t e = cudaSuccess;
  const int variant = p.q_out != nullptr ? 8 : p.b_mn_major ? 10 + (p.out_f32 ? 1 : 0)
                                                             : (p.b_row ? 4 : 0) + (p.out_f32 ? 2 : 0);
  switch (variant) {
#define FP8FG_VARIANT(V, R, F)                                                   \
  case V:                                                                        \
    kernels[0] = fp8_gemm_kernel<BN, R, F, kSplitNone, false, kVarPlain>;        \
    kernels[1] = fp8_gemm_kernel<BN, R, F, kSplitStream, false, kVarPlain>;      \
    kernels[2] = fp8_gemm_kernel<BN, R, F, kSplitNone, true, kVarPlain>;         \
    if constexpr (BN == 128) {                                                   \
      kernels[3] = fp8_gemm_kernel<BN, R, F, kSplitCluster, false, kVarPlain>;   \
      cluster_attr = ensure_smem_attr<BN, R, F, kSplitCluster, false>;           \
    }                                                                            \
    e = masked ? ensure_smem_attr<BN, R, F, kSplitNone, true>()                  \
               : ensure_smem_attr<BN, R, F, kSplitNone, false>();                \
    if (e == cudaSuccess && plan.sk) e = ensure_smem_attr<BN, R, F, kSplitStream, false>(); \
    break;
    FP8FG_VARIANT(0, false, false)
    FP8FG_VARIANT(2, false, true)
    FP8FG_VARIANT(4, true, false)
    FP8FG_VARIANT(6, true, true)
#undef FP8FG_VARIANT
    case 8:
      // fused 1x128 quantization of the BF16 output (dense, 128x256 tiles)
      if constexpr (BN == 256) {
        kernels[0] = fp8_gemm_kernel<BN, false, false, kSplitNone, false, kVarQuant>;
        kernels[1] = fp8_gemm_kernel<BN, false, false, kSplitStream, false, kVarQuant>;
        e = ensure_smem_attr<BN, false, false, kSplitNone, false, kVarQuant>();
        if (e == cudaSuccess && plan.sk) e = ensure_smem_attr<BN, false, false, kSplitStream, false, kVarQuant>();
      } else {
        e = cudaErrorInvalidValue;
      }
      break;
#define FP8FG_VARIANT_BT(V, F)                                                          \
  case V:                                                                               \
    if constexpr (BN != 192) {                                                          \
      kernels[0] = fp8_gemm_kernel<BN, false, F, kSplitNone, false, kVarBT>;            \
      kernels[1] = fp8_gemm_kernel<BN, false, F, kSplitStream, false, kVarBT>;          \
      if constexpr (BN == 128) {                                                        \
        kernels[3] = fp8_gemm_kernel<BN, false, F, kSplitCluster, false, kVarBT>;       \
        cluster_attr = ensure_smem_attr<BN, false, F, kSplitCluster, false, kVarBT>;    \
      }                                                                                 \
      e = ensure_smem_attr<BN, false, F, kSplitNone, false, kVarBT>();                  \
      if (e == cudaSuccess && plan.sk) e = ensure_smem_attr<BN, false, F, kSplitStream, false, kVarBT>(); \
    } else {                                                                            \
      e = cudaErrorInvalidValue;                                                        \
    }                                                                                   \
    break;
    // B read MN-major (the data-gradient GEMM), BF16 or FP32 out
    FP8FG_VARIANT_BT(10, false)
    FP8FG_VARIANT_BT(11, true)
#undef FP8FG_VARIANT_BT
    default:
      e = cudaErrorInvalidValue;
      break;
  }
  if (e != cudaSuccess) {
    *detail = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return e;
  }
  // the cluster split where it applies and the policy allows it
  int cl = 0;
  const int policy = split_policy();
  if (kernels[3] != nullptr && policy != kPolicyStream) {
    e = cluster_attr();
    if (e == cudaSuccess) e = pick_cluster_split(p.mode, p.rows, p.N, p.K, p.groups, num_sms, kernels[3], &cl);
    if (e != cudaSuccess) {
      *detail = "cluster split set-up (shared-memory attribute or cluster occupancy) failed";
      return e;
    }
  }
  // Automatic: the cluster split where it saves each CTA at least
  // kMinSavedBlocks K blocks (its reduction costs about that much: ~3 us
  // against ~0.33 us per 128-K block of the K loop, measured), whole tiles
  // where it applies but saves less (Stream-K's reduction costs more), and
  // Stream-K only where the cluster split does not apply.
  constexpr int64_t kMinSavedBlocks = 10;
  const bool cluster_pays = cl >= 2 && KB - (KB + cl - 1) / cl >= kMinSavedBlocks;
  const bool use_cluster = cl >= 2 && (policy == kPolicyCluster || (policy == kPolicyAuto && cluster_pays));
  const bool use_stream_k = plan.sk && !use_cluster && !(policy == kPolicyAuto && cl >= 2);
  if (use_cluster) {
    a.cl_split = cl;
    e = launch_kernel_cluster(kernels[3], dim3(static_cast<unsigned>(a.num_tiles * cl)), dim3(C::kThreads), C::kSmem,
                              stream, static_cast<unsigned>(cl), tmA, tmB, tmSA, tmSB, tmC, tmQ, a);
  } else if (!use_stream_k) {
    // whole tiles: one persistent CTA per SM at most
    const int grid = a.num_tiles < num_sms ? a.num_tiles : num_sms;
    e = launch_kernel(kernels[masked ? 2 : 0], dim3(grid), dim3(C::kThreads), C::kSmem, stream, tmA, tmB, tmSA, tmSB,
                      tmC, tmQ, a);
  } else {
    a.dp_tiles = plan.dp_tiles;
    a.sk_tile0 = plan.dp_tiles;
    a.sk_units = static_cast<int>(plan.sk_units);
    a.sk_per_cta = static_cast<int>(plan.sk_per_cta);
    a.sk_lcm = static_cast<int>(plan.sk_lcm);
    a.ws_count = static_cast<int*>(p.workspace);
    a.ws_partial = reinterpret_cast<float*>(static_cast<char*>(p.workspace) + plan.count_bytes);
    e = launch_kernel(kernels[1], dim3(plan.grid), dim3(C::kThreads), C::kSmem, stream, tmA, tmB, tmSA, tmSB, tmC, tmQ,
                      a);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) *detail = "GEMM kernel launch failed";
  return e;
}

// Tile width: FP8FG_BN=128|192|256 overrides (tuning). Otherwise 128 for
// dense problems of one 128-row block (decode): twice the tiles for
// Stream-K to spread the weight stream over, measured 25.2 -> 19.6 us at
// 128x4096x7168 and 37.4 -> 30.8 us at 64x7168x16384. 256 for the rest,
// where it is the fastest at every prefill and MoE shape measured.
int pick_bn(int mode, int64_t rows, bool quant_out = false) {
  if (quant_out) return 256;  // the fused quantization needs 128-column warps
  static int forced = [] {
    const char* v = std::getenv("FP8FG_BN");
    if (!v) return 0;
    const int b = std::atoi(v);
    return (b == 128 || b == 192 || b == 256) ? b : 0;
  }();
  if (forced) return forced;
  if (mode == kModeDense && rows <= BM) return 128;
  return 256;
}

}  // namespace

void set_split_policy(int policy) { g_split_policy.store(policy); }

namespace gemm_detail {

namespace {
constexpr int kMapCacheSize = 64;

struct MapCache {
  std::mutex mu;
  MapKey key[kMapCacheSize];
  MapSet maps[kMapCacheSize];
  int used = 0, next = 0;
};

MapCache& map_cache() {
  static MapCache c;
  return c;
}
}  // namespace

bool map_cache_find(const MapKey& k, MapSet* out) {
  MapCache& c = map_cache();
  std::lock_guard<std::mutex> lock(c.mu);
  for (int i = 0; i < c.used; ++i) {
    if (std::memcmp(&c.key[i], &k, sizeof(k)) == 0) {
      *out = c.maps[i];
      return true;
    }
  }
  return false;
}

void map_cache_put(const MapKey& k, const MapSet& m) {
  MapCache& c = map_cache();
  std::lock_guard<std::mutex> lock(c.mu);
  const int slot = c.used < kMapCacheSize ? c.used++ : c.next;
  c.next = (slot + 1) % kMapCacheSize;
  c.key[slot] = k;
  c.maps[slot] = m;
}

}  // namespace gemm_detail

size_t gemm_workspace_bytes(int mode, int64_t rows, int64_t N, int64_t K, int64_t groups, int num_sms) {
  // enough for the plain and the fused-quantization tile choice of the shape
  size_t need = 0;
  for (bool q : {false, true}) {
    const Plan plan = plan_gemm(mode, rows, N, K, groups, num_sms, pick_bn(mode, rows, q), SIZE_MAX);
    if (plan.sk && plan.partial_bytes + plan.count_bytes > need) need = plan.partial_bytes + plan.count_bytes;
  }
  return need;
}

void gemm_workspace_zero_range(int mode, int64_t rows, int64_t N, int64_t K, int64_t groups, int num_sms,
                               size_t workspace_bytes, size_t* offset, size_t* bytes) {
  const Plan plan = plan_gemm(mode, rows, N, K, groups, num_sms, pick_bn(mode, rows), workspace_bytes);
  *offset = 0;
  *bytes = plan.sk ? plan.count_bytes : 0;
}

cudaError_t launch_gemm(const GemmProblem& p, uint32_t* status, uint64_t wait_limit_ns, int debug_skip_fill,
                        int num_sms, cudaStream_t stream, const char** detail) {
  if (bs_gemm_eligible(p)) return launch_gemm_bs(p, status, wait_limit_ns, debug_skip_fill, num_sms, stream, detail);
  if (p.q_out == nullptr && !p.b_mn_major && pair_gemm_eligible(p, num_sms))
    return launch_gemm_pair(p, status, wait_limit_ns, debug_skip_fill, stream, detail);
  int bn = pick_bn(p.mode, p.rows, p.q_out != nullptr);
  if (p.b_mn_major && bn == 192) bn = 256;
  switch (bn) {
    case 192: return launch_bn<192>(p, status, wait_limit_ns, debug_skip_fill, num_sms, stream, detail);
    case 256: return launch_bn<256>(p, status, wait_limit_ns, debug_skip_fill, num_sms, stream, detail);
    default: return launch_bn<128>(p, status, wait_limit_ns, debug_skip_fill, num_sms, stream, detail);
  }
}

}  // namespace fp8fg
