// FP8 GEMM with fine-grained scaling on CTA pairs (tcgen05 cta_group::2),
// for dense problems with enough rows to fill 256-row tiles.
//
// What it computes is what gemm.cu computes (DeepSeek-V3 report excerpt,
// page 1, paragraph 3): per 128-wide K block the FP8 partial sums are
// promoted to FP32 registers, scaled by sA[m, kb] * sB[n, kb], and
// accumulated in FP32; the output is BF16 or FP32.
//
// Why pairs. One CTA computing a 128 x 256 tile reads its A and B operands
// from shared memory for every MMA and has TMA write them there: for every
// 128-K block about 96 KB pass through that SM's shared memory. With
// cta_group::2 the two CTAs of a cluster compute one 256 x 256 tile: each
// loads its own 128 rows of A and half of the tile's B (128 rows), and the
// tensor cores of the pair share the B halves, so every SM moves 64 KB per
// K block. Measured on B300 (4096 x N x 7168, BF16 out): level with the
// single-CTA kernel under sustained, power-capped load (+2.5% at N=24576,
// where the lower operand traffic lets the clock sit higher), 2-4% behind
// it in short bursts. So it is an option (fp8fg_debug_set key 3), not the
// default.
//
// Roles (each CTA, 10 warps):
//   warp 0     TMA producer: this CTA's A rows and B half into a 5-stage
//              ring. A and B completions count on the LEADER's full barrier
//              (both CTAs' bytes); the scales land on a local barrier.
//   warp 1     leader only: MMA issuer. Per K block: wait for an
//              accumulator buffer released by the promotion warps of both
//              CTAs, issue 4 x tcgen05.mma.cta_group::2 (M 256, N 256,
//              K 32), commit to the buffer's "full" barrier in both CTAs.
//   warps 2-9  promotion + epilogue. Warp w reads TMEM lanes 32*(w%4)...
//              (its rows) and the 128 columns of its column group g: tile
//              columns 128*g .. 128*g+127, inside one 128x128 block of B
//              scales. acc += (sA * sB) * partial per K block, then the tile
//              is stored through shared-memory staging and TMA stores.
// TMEM column c of a buffer holds tile column c: the MMA takes B rows
// 0..N/2-1 from the leader's shared memory and the rest from the peer's.
// (With two groups, column c of group h's buffer holds tile column
// 64*h + c for c < 64 and 128 + 64*h + (c - 64) otherwise.)
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"
#include "launch.h"
#include "tmap.h"

namespace fp8fg {

namespace {

using namespace gemm_detail;

struct PairCfg {
  static constexpr int kStages = 5;
  static constexpr int kTileM = 2 * BM;   // rows of a pair tile
  static constexpr int kTileN = 256;      // columns of a pair tile
  // MMA groups per K block: 1 = one N=256 group into a 256-column buffer
  // (two in TMEM); 2 = two N=128 groups into 128-column buffers (four).
  // Two groups halve the MMA work per instruction, and one issuing thread
  // (about 30-50 ns per tcgen05.mma next to busy promotion warps) then
  // bounds the K block: measured 20-25% slower than one group, and still
  // 10% slower with the groups split over two issuing threads.
  static constexpr int kGroups = 1;
  static constexpr int kHalfCols = kTileN / kGroups;  // TMEM columns of one buffer (MMA N)
  static constexpr int kHalfBufs = 512 / kHalfCols;
  static constexpr int kGroupRows = (kTileN / 2) / kGroups;  // B rows of each CTA per group
  static constexpr int kTmemCols = 512;
  // MMA-issuing threads (leader, lane 0 of warps 1 .. kIssuers): issuer i
  // takes the groups h with h % kIssuers == i
  static constexpr int kIssuers = 1;
  static constexpr int kEpiWarps = 8;
  static constexpr int kEpiWarp0 = kIssuers > 1 ? 4 : 2;
  static constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;  // 168 registers a thread either way
  static constexpr int kNC = 128;                                 // accumulator columns per thread
  static constexpr int kABytes = BM * BK;                         // this CTA's 128 rows of A
  static constexpr int kBBytes = (kTileN / 2) * BK;               // this CTA's half of B
  static constexpr int kSABytes = BM * 4;
  static constexpr int kSBBytes = kTileN * 4;                     // per-row B scales, whole tile
  static constexpr int kEpiWarpBytes = 32 * kNC * 2;              // 8 KB staging per warp
  static constexpr int kBorrowWarps = (kABytes + kBBytes) / kEpiWarpBytes;  // 4
  static constexpr int kEpiBytes = (kEpiWarps - kBorrowWarps) * kEpiWarpBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffEpi = kOffB + kStages * kBBytes;
  static constexpr int kOffSA = kOffEpi + kEpiBytes;
  static constexpr int kOffSB = kOffSA + kStages * kSABytes;
  static constexpr int kOffSbw = kOffSB + kStages * kSBBytes;
  static constexpr int kSbwChunk = 128;
  static constexpr int kOffBar = kOffSbw + kEpiWarps * kSbwChunk * 4;
  // full[S] (leader: A and B of both CTAs), sfull[S] (scales), empty[S],
  // tfull[4], tempty[4] (leader: 2 x 8 promotion warps), drain
  static constexpr int kNumBars = 3 * kStages + 2 * kHalfBufs + kIssuers;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffTmemSlot + 16 + 1024;
  static_assert(kHalfBufs * kHalfCols == kTmemCols, "half buffers fill TMEM");
  static_assert(kSmem > 116 * 1024, "one CTA per SM: the TMEM allocation never waits on a neighbour");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert((kOffB % 1024) == 0 && (kOffEpi % 1024) == 0 && (kABytes % 1024) == 0,
                "128-byte swizzled tiles need 1024-byte alignment");
};

template <bool kBRow, bool kF32>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg::kThreads, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                         const __grid_constant__ CUtensorMap tmC, const KArgs a) {
  using C = PairCfg;
  constexpr int S = C::kStages;
  constexpr int NB = C::kHalfBufs;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());

  const uint32_t bar0 = sbase + C::kOffBar;
  auto full_bar = [bar0](uint32_t s) { return bar0 + s * 8; };
  auto sfull_bar = [bar0](uint32_t s) { return bar0 + (S + s) * 8; };
  auto empty_bar = [bar0](uint32_t s) { return bar0 + (2 * S + s) * 8; };
  auto tfull_bar = [bar0](uint32_t b) { return bar0 + (3 * S + b) * 8; };
  auto tempty_bar = [bar0](uint32_t b) { return bar0 + (3 * S + NB + b) * 8; };
  auto drain_bar = [bar0](uint32_t i) { return bar0 + (3 * S + 2 * NB + i) * 8; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSA);
    if (kBRow) prefetch_tmap(&tmSB);
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(sfull_bar(s), 1);
      mbar_init(empty_bar(s), C::kEpiWarps);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * C::kEpiWarps);
    }
    for (int i = 0; i < C::kIssuers; ++i) mbar_init(drain_bar(i), 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);  // both CTAs
  tc_fence_before();
  // both CTAs' barriers exist and TMEM is allocated before any cross-CTA
  // arrival, TMA completion or MMA
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  grid_dependency_sync();

  const int tiles_m = a.tiles_m;  // pair-tile rows: ceil(M / 256)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t full_leader = map_to_cta(full_bar(0), 0);
      constexpr uint32_t tx_ab = C::kABytes + C::kBBytes;
      constexpr uint32_t tx_scales = C::kSABytes + (kBRow ? C::kSBBytes : 0);
      uint32_t it = 0;
      bool ok = true;
      for (int t = pair; ok && t < a.num_tiles; t += npairs) {
        const int m0 = (t % tiles_m) * C::kTileM + static_cast<int>(rank) * BM;
        const int n0 = (t / tiles_m) * C::kTileN;
        const int nb0 = n0 + static_cast<int>(rank) * (C::kTileN / 2);
        for (int kb = 0; kb < a.KB; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1;
          if (!mbar_wait(empty_bar(s), ph ^ 1, a.status, kStatusTimeoutProducer, a.wait_limit_ns)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * tx_ab);
          mbar_arrive_expect_tx(sfull_bar(s), tx_scales);
          if (static_cast<int>(it) == a.debug_skip_fill) continue;  // test hook: never filled
          tma_load_3d_pair(sbase + C::kOffA + s * C::kABytes, &tmA, full_leader + s * 8, kb * BK, m0, 0);
          tma_load_3d_pair(sbase + C::kOffB + s * C::kBBytes, &tmB, full_leader + s * 8, kb * BK, nb0, 0);
          tma_load_3d(sbase + C::kOffSA + s * C::kSABytes, &tmSA, sfull_bar(s), m0, kb, 0);
          if (kBRow) tma_load_3d(sbase + C::kOffSB + s * C::kSBBytes, &tmSB, sfull_bar(s), n0, kb, 0);
        }
      }
      // No copy may still be landing when the CTA exits: wait (bounded,
      // ignoring the error word) for the last fill of each stage. The leader's
      // full barrier also counts the peer's A and B bytes.
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
      for (uint32_t i = first; i < it; ++i) {
        mbar_wait(sfull_bar(i % S), (i / S) & 1, nullptr, 0, a.wait_limit_ns);
        if (leader) mbar_wait(full_bar(i % S), (i / S) & 1, nullptr, 0, a.wait_limit_ns);
      }
    }
  } else if (warp < C::kEpiWarp0) {
    // ------------------------------------------------------------ MMA issuers (leader)
    const int issuer = warp - 1;
    if (leader && lane == 0 && issuer < C::kIssuers) {
      constexpr uint32_t idesc = f8_idesc(C::kTileM, C::kHalfCols);
      uint32_t it = 0;
      bool ok = true;
      for (int t = pair; ok && t < a.num_tiles; t += npairs) {
        for (int kb = 0; kb < a.KB && ok; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1;
          if (!mbar_wait(full_bar(s), ph, a.status, kStatusTimeoutMma, a.wait_limit_ns)) {
            ok = false;
            break;
          }
          const uint64_t ad = kmajor_sw128_desc(sbase + C::kOffA + s * C::kABytes);
#pragma unroll
          for (int h = issuer; h < C::kGroups; h += C::kIssuers) {
            const uint32_t u = C::kGroups * it + h;
            const uint32_t b = u % NB, tph = (u / NB) & 1;
            if (!mbar_wait(tempty_bar(b), tph ^ 1, a.status, kStatusTimeoutMma, a.wait_limit_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // the group's rows of each CTA's B half (whole 1 KB swizzle atoms)
            const uint64_t bd = kmajor_sw128_desc(sbase + C::kOffB + s * C::kBBytes + h * C::kGroupRows * BK);
            const uint32_t d = tmem_base + b * C::kHalfCols;
#pragma unroll
            for (int k = 0; k < BK / 32; ++k) mma_f8f6f4_pair(d, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
            mma_commit_pair(tfull_bar(b), 0x3);
          }
        }
      }
      // All MMAs of this issuer complete before TMEM is released.
      mma_commit_pair(drain_bar(issuer), 0x1);
      if (!mbar_wait(drain_bar(issuer), 0, nullptr, 0, a.wait_limit_ns)) atomicCAS(a.status, 0u, kStatusTimeoutDrain);
    }
  } else {
    // ------------------------------------------------------------ promotion + epilogue
    constexpr int NC = C::kNC;
    const int ew = warp - C::kEpiWarp0;
    const int quarter = warp & 3;             // TMEM lanes this warp may access
    const int g = ew >> 2;                    // column group: tile columns 128g .. 128g+127
    const int col0 = g * 128;
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tempty_leader = map_to_cta(tempty_bar(0), 0);
    const float* smem_sa = reinterpret_cast<const float*>(smem + C::kOffSA);
    const float* smem_sb = reinterpret_cast<const float*>(smem + C::kOffSB);
    float* sbw = reinterpret_cast<float*>(smem + C::kOffSbw) + ew * C::kSbwChunk;
    float acc[NC];
    uint32_t it = 0;
    bool ok = true;
    int held = -1;
    for (int t = pair; ok && t < a.num_tiles; t += npairs) {
      Tile ti;
      ti.m0 = (t % tiles_m) * C::kTileM + static_cast<int>(rank) * BM;
      ti.n0 = (t / tiles_m) * C::kTileN;
      ti.gA = ti.gB = ti.gC = 0;
      ti.kb0 = 0;
      ti.kbc = a.KB;
      ti.tile = t;
      ti.sk_start = -1;
      ti.skip = false;
#pragma unroll
      for (int j = 0; j < NC; ++j) acc[j] = 0.0f;
      for (unsigned jb = 0; jb < static_cast<unsigned>(a.KB); ++jb, ++it) {
        const uint32_t s = it % S, ph = (it / S) & 1;
        if (!kBRow && (jb % C::kSbwChunk) == 0) {
          const int nbk = (ti.n0 + col0) / 128;
          const float* src = a.sB + static_cast<int64_t>(nbk) * a.sb_kblk;
          __syncwarp();
#pragma unroll
          for (int i = 0; i < C::kSbwChunk / 32; ++i) {
            const unsigned k = jb + i * 32 + lane;
            sbw[i * 32 + lane] = (nbk < a.sb_nblk && k < static_cast<unsigned>(a.KB)) ? __ldg(src + k) : 0.0f;
          }
          __syncwarp();
        }
        const bool got_s = mbar_wait(sfull_bar(s), ph, a.status, kStatusTimeoutEpilogue, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, got_s)) {
          ok = false;
          break;
        }
        const float sa = smem_sa[s * BM + row_in_tile];
        float sc = 0.0f;
        if constexpr (!kBRow) sc = sa * sbw[jb % C::kSbwChunk];
        const float* sbv = smem_sb + s * C::kTileN + col0;
#pragma unroll
        for (int h = 0; h < C::kGroups; ++h) {
          const uint32_t u = C::kGroups * it + h;
          const uint32_t b = u % NB, tph = (u / NB) & 1;
          const bool got = mbar_wait(tfull_bar(b), tph, a.status, kStatusTimeoutEpilogue, a.wait_limit_ns);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + lane_bits + b * C::kHalfCols + g * C::kGroupRows;
#pragma unroll
          for (int ch = 0; ch < C::kGroupRows / 16; ++ch) {
            uint32_t r[16];
            tmem_ld16(taddr + ch * 16, r);
            promote<16, kBRow>(acc + h * C::kGroupRows + ch * 16, r, sc, sa, sbv + h * C::kGroupRows + ch * 16);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader)
              mbar_arrive(tempty_bar(b));
            else
              mbar_arrive_remote(tempty_leader + b * 8);
          }
        }
        if (!ok) break;
        // the staging warps keep the tile's last stage for the epilogue
        const bool hold = ew < C::kBorrowWarps && jb + 1 == static_cast<unsigned>(a.KB);
        if (hold) held = static_cast<int>(s);
        if (lane == 0 && !hold) mbar_arrive(empty_bar(s));
      }
      if (!ok) break;
      bool staged = false;
      uint8_t* region;
      if (held >= 0 && ew < 2)
        region = smem + C::kOffA + held * C::kABytes + ew * C::kEpiWarpBytes;
      else if (held >= 0)
        region = smem + C::kOffB + held * C::kBBytes + (ew - 2) * C::kEpiWarpBytes;
      else
        region = smem + C::kOffEpi + (ew - C::kBorrowWarps) * C::kEpiWarpBytes;  // ew >= kBorrowWarps here
      staged = store_tile_tma<NC, kF32>(a, ti, row_in_tile, col0, lane, region, &tmC, acc);
      if (!staged) store_row<NC, kF32>(a, ti, row_in_tile, col0, acc);
      if (held >= 0) {
        if (lane == 0) {
          if (staged) bulk_wait_read_all();
          mbar_arrive(empty_bar(held));
        }
        held = -1;
      }
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  // Both CTAs are done with TMEM (the leader has drained its MMAs) before
  // either releases it. After an expired wait, copies of the peer may still
  // be in flight toward the leader's barriers: give them 100 us to land
  // before this CTA's shared memory goes away.
  cluster_sync();
  if (*reinterpret_cast<volatile uint32_t*>(a.status) != 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
bool encode_pair_maps(const GemmProblem& p, MapSet* m) {
  using C = PairCfg;
  const int64_t KB = p.K / BK;
  bool ok = make_map(&m->a, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.A, p.K, p.rows, 1, p.K, p.rows * p.K, BK, BM,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&m->b, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.B, p.K, p.N, 1, p.K, p.N * p.K, BK, C::kTileN / 2,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&m->sa, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.sA, p.rows, KB, 1, ld4(p.rows) * 4,
                      KB * ld4(p.rows) * 4, BM, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (p.b_row) {
    ok = ok && make_map(&m->sb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.sB, p.N, KB, 1, ld4(p.N) * 4, KB * ld4(p.N) * 4,
                        C::kTileN, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    m->sb = m->sa;  // unused
  }
  const int64_t esz = p.out_f32 ? 4 : 2;
  ok = ok && make_map(&m->c, p.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.C,
                      p.N, p.rows, 1, p.N * esz, p.rows * p.N * esz, 128 / esz, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  return ok;
}

template <bool kBRow, bool kF32>
cudaError_t pair_setup(int* max_pairs) {
  // per device: the shared-memory limit and the number of clusters of two
  // that fit at once (every pair needs two SMs of one TPC)
  static std::atomic<int> pairs[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int v = pairs[dev & 63].load(std::memory_order_acquire);
  if (v > 0) {
    *max_pairs = v;
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(fp8_gemm_pair_kernel<kBRow, kF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PairCfg::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(PairCfg::kThreads);
  cfg.dynamicSmemBytes = PairCfg::kSmem;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, fp8_gemm_pair_kernel<kBRow, kF32>, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  pairs[dev & 63].store(clusters, std::memory_order_release);
  *max_pairs = clusters;
  return cudaSuccess;
}

}  // namespace

namespace {
// Off by default; FP8FG_PAIR=1 in the environment, or fp8fg_debug_set(3, 1),
// sends large dense problems to the pair kernel.
std::atomic<int> g_pair_enabled{[] {
  const char* v = std::getenv("FP8FG_PAIR");
  return (v && v[0] == '1') ? 1 : 0;
}()};
}  // namespace

void set_pair_gemm_enabled(bool on) { g_pair_enabled.store(on ? 1 : 0); }

bool pair_gemm_eligible(const GemmProblem& p, int num_sms) {
  const bool enabled = g_pair_enabled.load() != 0;
  // Dense problems whose 128 x 256 tiles outnumber half the SMs (fewer go
  // to the single-CTA kernel, which splits K over the idle SMs), with at
  // least one whole 256 x 256 pair tile.
  const int64_t tiles = ((p.rows + BM - 1) / BM) * ((p.N + 255) / 256);
  return enabled && p.mode == kModeDense && p.rows >= PairCfg::kTileM && p.N >= PairCfg::kTileN &&
         tiles * 2 > num_sms;
}

cudaError_t launch_gemm_pair(const GemmProblem& p, uint32_t* status, uint64_t wait_limit_ns, int debug_skip_fill,
                             cudaStream_t stream, const char** detail) {
  using C = PairCfg;
  MapKey k;
  std::memset(&k, 0, sizeof(k));
  k.A = p.A; k.B = p.B; k.sA = p.sA; k.sB = p.b_row ? p.sB : nullptr; k.C = p.C;
  k.rows = p.rows; k.N = p.N; k.K = p.K; k.groupsA = 1; k.groupsB = 1; k.groupsC = 1;
  k.kind = -2; k.b_row = p.b_row; k.out_f32 = p.out_f32;
  MapSet ms;
  if (!map_cache_find(k, &ms)) {
    if (!encode_pair_maps(p, &ms)) {
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
  a.tiles_m = static_cast<int>((p.rows + C::kTileM - 1) / C::kTileM);
  a.tiles_n = static_cast<int>((p.N + C::kTileN - 1) / C::kTileN);
  const int64_t nt = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  if (nt > 0x7FFFFFFF) {
    *detail = "too many output tiles";
    return cudaErrorInvalidValue;
  }
  a.num_tiles = static_cast<int>(nt);
  a.groupsB = 1;
  a.accumulate = p.accumulate;
  a.sB = p.sB;
  a.sb_nblk = static_cast<int>((p.N + 127) / 128);
  a.sb_kblk = a.KB;
  a.C = p.C;
  a.ldc = p.N;
  a.c_group_stride = p.rows * p.N;
  a.status = status;
  a.wait_limit_ns = wait_limit_ns;
  a.debug_skip_fill = debug_skip_fill;
  a.dp_tiles = a.num_tiles;
  using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, KArgs);
  KernelFn fn = nullptr;
  int max_pairs = 0;
  cudaError_t e = cudaSuccess;
  switch ((p.b_row ? 2 : 0) + (p.out_f32 ? 1 : 0)) {
    case 0: fn = fp8_gemm_pair_kernel<false, false>; e = pair_setup<false, false>(&max_pairs); break;
    case 1: fn = fp8_gemm_pair_kernel<false, true>; e = pair_setup<false, true>(&max_pairs); break;
    case 2: fn = fp8_gemm_pair_kernel<true, false>; e = pair_setup<true, false>(&max_pairs); break;
    default: fn = fp8_gemm_pair_kernel<true, true>; e = pair_setup<true, true>(&max_pairs); break;
  }
  if (e != cudaSuccess) {
    *detail = "pair kernel set-up (shared-memory attribute or cluster occupancy) failed";
    return e;
  }
  const int pairs = a.num_tiles < max_pairs ? a.num_tiles : max_pairs;
  e = launch_kernel(fn, dim3(2 * pairs), dim3(C::kThreads), C::kSmem, stream, ms.a, ms.b, ms.sa, ms.sb, ms.c, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) *detail = "pair GEMM kernel launch failed";
  return e;
}

}  // namespace fp8fg
