// Pieces shared by the GEMM kernels (gemm.cu: one CTA per output tile;
// gemm_pair.cu: CTA pairs on one tile with tcgen05 cta_group::2): the
// kernel arguments, the output-tile descriptor, the FP32 promotion step, the
// epilogue stores, and the host-side cache of tensor maps.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace fp8fg {
namespace gemm_detail {

constexpr int BM = 128;  // rows of an output tile per CTA (TMEM lanes)
constexpr int BK = 128;  // K block: one scale block, one promotion

struct KArgs {
  int mode;
  int rows, N, K;
  int tiles_m, tiles_n, num_tiles;
  int groupsB;
  int accumulate;
  const int32_t* m_indices;
  const int32_t* masked;
  const float* sB;
  int sb_nblk, sb_kblk;
  // block scale of output-column block nb and K block kb of group g:
  // sB[(g * sb_nblk * sb_kblk) + nb * sb_col_stride + kb * sb_red_stride]
  // ([nb][kb] for weights quantized as B; [kb][nb], transposed, when the
  // weight is read as its own transpose in the data-gradient GEMM)
  int sb_col_stride, sb_red_stride;
  void* C;
  int64_t ldc;
  int64_t c_group_stride;
  uint32_t* status;
  uint64_t wait_limit_ns;
  int debug_skip_fill;
  // Stream-K (dense only, the kSplit variant): tiles [0, dp_tiles) run
  // whole, tile t on CTA t % gridDim.x; the K blocks of tiles sk_tile0 ..
  // are sk_units "units" in tile-major order and CTA c takes units
  // [c * sk_per_cta, (c + 1) * sk_per_cta). A tile whose units fall to
  // several CTAs is summed, in piece order, by the last piece to arrive,
  // from FP32 partials in ws_partial (one slot per segment, see reduce_sk).
  int KB;
  int dp_tiles;
  int sk_tile0;                      // first split tile (the tiles before it run whole)
  int sk_units, sk_per_cta, sk_lcm;  // the planner keeps them below 2^31
  float* ws_partial;
  int* ws_count;
  // Cluster split (dense, the kSplitCluster variant): tile t is computed by
  // the cl_split CTAs of cluster t, CTA r of it taking K blocks
  // [r * KB / cl_split, (r + 1) * KB / cl_split); the partial sums meet in
  // shared memory (see cluster_reduce_store).
  int cl_split;
  // rows of A one TMA fill loads (a_box_rows(rows), see there)
  int a_rows_box;
  // MMA issuer warps (1 or 2): issuer i takes the K blocks it % n == i
  int mma_issuers;
  // fused 1x128 quantization of the BF16 output (the kQ kernel variant)
  float* s_out;
  int64_t ld_s;
  int pow2_out;
  int c_bf16;  // the BF16 C is stored as well
};

struct Tile {
  int gA, gB, gC, m0, n0, kb0, kbc, tile;
  int sk_start;  // Stream-K segment: its first unit; -1 for a whole tile
  bool skip;
};

// Convert and store one epilogue thread's share of a tile row.
template <int NC, bool kF32>
__device__ __forceinline__ void store_row(const KArgs& a, const Tile& ti, int row_in_tile, int col0,
                                          const float (&acc)[NC]) {
  const int row = ti.m0 + row_in_tile;
  if (row >= a.rows) return;
  if (a.mode == kModeContig && __ldg(a.m_indices + row) < 0) return;
  if (a.mode == kModeMaskedRows && row >= __ldg(a.masked + ti.gC)) return;
  const int ncol = a.N - (ti.n0 + col0);  // a multiple of 8 (N % 8 == 0)
  const int64_t off = static_cast<int64_t>(ti.gC) * a.c_group_stride + static_cast<int64_t>(row) * a.ldc +
                      ti.n0 + col0;
  if constexpr (kF32) {
    float* c = static_cast<float*>(a.C) + off;
#pragma unroll
    for (int j = 0; j < NC; j += 4) {
      if (j < ncol) {
        float4 v = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
        if (a.accumulate) {
          const float4 o = *reinterpret_cast<const float4*>(c + j);
          v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
        }
        *reinterpret_cast<float4*>(c + j) = v;
      }
    }
  } else {
    __nv_bfloat16* c = static_cast<__nv_bfloat16*>(a.C) + off;
#pragma unroll
    for (int j = 0; j < NC; j += 8) {
      if (j < ncol) {
        uint4 v;
        v.x = pack_bf16x2(acc[j], acc[j + 1]);
        v.y = pack_bf16x2(acc[j + 2], acc[j + 3]);
        v.z = pack_bf16x2(acc[j + 4], acc[j + 5]);
        v.w = pack_bf16x2(acc[j + 6], acc[j + 7]);
        *reinterpret_cast<uint4*>(c + j) = v;
      }
    }
  }
}

// Tile rows of one epilogue warp (32 rows x NC columns) through its 8 KB
// shared-memory staging area and TMA stores, when every row of the warp may
// be written (dense: rows past M are clipped by the tensor map; grouped
// layouts: no padding or masked rows among the 32). Returns false, having
// done nothing, otherwise; the caller then stores row by row.
// Staging: two boxes of 32 rows x 128 bytes (BF16: 64 columns each; FP32:
// 32 columns each, so FP32 goes out in two rounds of 64 columns) with the
// 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r % 8)): a warp's
// 16-byte writes of one chunk index hit 8 distinct chunks, conflict free.
// FP32 with accumulate adds into C with the TMA reduce-add.
template <int NC, bool kF32>
__device__ __forceinline__ bool store_tile_tma(const KArgs& a, const Tile& ti, int row_in_tile, int col0, int lane,
                                               uint8_t* region, const CUtensorMap* tmC, const float (&acc)[NC]) {
  const int row = ti.m0 + row_in_tile;
  bool ok = true;
  if (a.mode == kModeContig) ok = row < a.rows && __ldg(a.m_indices + row) >= 0;
  if (a.mode == kModeMaskedRows) ok = row < __ldg(a.masked + ti.gC);
  if (!__all_sync(0xffffffffu, ok)) return false;
  constexpr int kColsPerRound = 64;          // two 128-byte boxes
  constexpr int kBoxCols = kF32 ? 32 : 64;
  const int y = ti.m0 + (row_in_tile & ~31);
#pragma unroll
  for (int rd = 0; rd < NC / kColsPerRound; rd += (kF32 ? 1 : 2)) {
    // the previous stores must have read the staging area, and the tensor
    // core's reads of a borrowed stage come before these writes
    if (lane == 0) bulk_wait_read_all();
    fence_async_shared();
    __syncwarp();
#pragma unroll
    for (int b = 0; b < 2; ++b) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 v;
        if constexpr (kF32) {
          const int j = rd * kColsPerRound + b * kBoxCols + c * 4;
          v = make_uint4(__float_as_uint(acc[j]), __float_as_uint(acc[j + 1]), __float_as_uint(acc[j + 2]),
                         __float_as_uint(acc[j + 3]));
        } else {
          const int j = b * kBoxCols + c * 8;
          v.x = pack_bf16x2(acc[j], acc[j + 1]);
          v.y = pack_bf16x2(acc[j + 2], acc[j + 3]);
          v.z = pack_bf16x2(acc[j + 4], acc[j + 5]);
          v.w = pack_bf16x2(acc[j + 6], acc[j + 7]);
        }
        *reinterpret_cast<uint4*>(region + b * 4096 + lane * 128 + ((c ^ (lane & 7)) << 4)) = v;
      }
    }
    fence_async_shared();
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int x = ti.n0 + col0 + (kF32 ? rd * kColsPerRound : 0) + b * kBoxCols;
        if (kF32 && a.accumulate)
          tma_reduce_add_3d(tmC, smem_u32(region + b * 4096), x, y, ti.gC);
        else
          tma_store_3d(tmC, smem_u32(region + b * 4096), x, y, ti.gC);
      }
      bulk_commit();
    }
  }
  return true;
}

// acc[j] += partial[j] * sc  (block-scaled B)   or
// acc[j] += partial[j] * sbv[j] * sa            (per-row B scales)
template <int W, bool kBRow>
__device__ __forceinline__ void promote(float* acc, const uint32_t (&r)[W], float sc, float sa, const float* sbv) {
  // Pairs of columns on the packed f32x2 pipe: each element still gets one
  // IEEE round-to-nearest FMA (and, for per-row B scales, one multiply).
#pragma unroll
  for (int j = 0; j < W; j += 2) {
    const uint64_t p = pk2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
    uint64_t a2 = pk2(acc[j], acc[j + 1]);
    if constexpr (kBRow) {
      const float2 b = *reinterpret_cast<const float2*>(sbv + j);
      a2 = fma2(mul2(p, pk2(b.x, b.y)), pk2(sa, sa), a2);
    } else {
      a2 = fma2(p, pk2(sc, sc), a2);
    }
    const float2 f = unpk2(a2);
    acc[j] = f.x;
    acc[j + 1] = f.y;
  }
}

// ---------------------------------------------------------------- host side
inline int64_t ld4(int64_t r) { return (r + 3) / 4 * 4; }

// Rows of A that one fill of a pipeline stage loads. A problem of one row
// tile (fewer than BM rows, as in decoding) loads only its rows, rounded up
// to the 8-row swizzle atom, instead of a full box whose rows past the end
// the copy engine would fill with zeros: at 64 rows that is a quarter of
// each stage's bytes. The MMA still runs 128 rows; the rows past the box
// hold stale shared memory, which reaches only accumulator rows that are
// never stored (row m of A B^T depends on row m of A alone).
inline int a_box_rows(int64_t rows) { return rows < BM ? static_cast<int>((rows + 7) / 8 * 8) : BM; }

// Tensor maps of one launch. Encoding them costs host time on every call,
// and a map depends only on the pointers and sizes in the key, so launches
// look them up in a small cache keyed by exactly those fields (a map for a
// freed and reused address with the same sizes is still the right map).
struct MapKey {
  const void* A;
  const void* B;
  const void* sA;
  const void* sB;
  const void* C;
  const void* Q;
  int64_t rows, N, K, groupsA, groupsB, groupsC;
  int32_t kind, b_row, out_f32, pad;  // kind: tile configuration of the launch
};

struct MapSet {
  CUtensorMap a, b, sa, sb, c, q;
};

// Thread-safe lookup / insertion (gemm.cu); a lookup that misses returns false.
bool map_cache_find(const MapKey& k, MapSet* out);
void map_cache_put(const MapKey& k, const MapSet& m);

}  // namespace gemm_detail
}  // namespace fp8fg
