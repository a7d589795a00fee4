// Internal launchers (host side); the public C ABI lives in include/fp8fg.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8fg {

// Launch context shared by the quantizer launchers: SM count (grid size),
// the device status word that receives timeout codes, the bounded-wait limit
// and the test hook that makes a producer skip one of its fills (-1: off).
struct QuantLaunch {
  int num_sms;
  uint32_t* status;
  uint64_t wait_limit_ns;
  int debug_skip_fill;
};

cudaError_t launch_quant_1x128(const void* x, bool f32, int64_t M, int64_t K, int64_t ldx, uint8_t* q, float* s,
                               int64_t lds, int pow2, const QuantLaunch& l, cudaStream_t stream);

cudaError_t launch_quant_128x128(const void* w, bool f32, int64_t G, int64_t N, int64_t K, uint8_t* q, float* s,
                                 int pow2, const QuantLaunch& l, cudaStream_t stream);

// src_kind: 0 E4M3 (+ s_src with row stride ld_t), 1 BF16, 2 FP32
cudaError_t launch_requant_128x1(const void* src, int src_kind, const float* s_src, int64_t ld_t, int64_t G,
                                 int64_t T, int64_t C, const int32_t* valid_rows, uint8_t* qT, float* sT,
                                 int64_t ld_c, int pow2, const QuantLaunch& l, cudaStream_t stream);

// Scheduling modes of the GEMM kernel.
enum GemmMode : int { kModeDense = 0, kModeContig = 1, kModeMaskedRows = 2, kModeMaskedK = 3 };

struct GemmProblem {
  int mode;
  const uint8_t* A;      // [groupsA][rows][K]
  const float* sA;       // [groupsA][K/128][ld(rows)]
  const uint8_t* B;      // [groupsB][N][K]
  const float* sB;       // block: [groupsB][ceil(N/128)][K/128]; row: [groupsB][K/128][ld(N)]
  int b_row;             // 1: per-row (128x1) B scales
  int b_mn_major;        // 1: B given as [K][N] (N contiguous), block scales [K/128][ceil(N/128)]
  int b_scale_pow2;      // 1 (with b_row): both operands' row scales are powers of two
  void* C;               // [groupsC][rows][N]
  int out_f32;
  int accumulate;
  int64_t rows;          // rows of A (and C) per group
  int64_t N, K;
  int64_t groups;        // groups of tiles (masked modes: E; otherwise 1)
  int64_t groupsB;       // groups of B (contig: E; masked: E; dense: 1)
  const int32_t* m_indices;
  const int32_t* masked;
  void* workspace;          // Stream-K scratch (zeroed before first use), or nullptr
  size_t workspace_bytes;
  // Fused quantization of the output (dense only; C, if not null, is BF16):
  // the BF16-rounded C quantized per 1x128 tile to E4M3 codes q_out [rows][N]
  // and scales s_out [N/128][ld(rows)]. q_out == nullptr: no quantization.
  uint8_t* q_out;
  float* s_out;
  int pow2_out;
};

// Bytes of Stream-K workspace launch_gemm uses for this problem when given
// enough (0: the problem is not split).
size_t gemm_workspace_bytes(int mode, int64_t rows, int64_t N, int64_t K, int64_t groups, int num_sms);

// Record the calling thread's last error message (fp8fg_last_error_string).
void set_last_error(const char* msg);

// Host-side argument checks shared by the dense GEMM entry points (sizes,
// enums, null pointers, alignment). Returns FP8FG_OK or an FP8FG_ERR_* code
// with the message recorded; never touches the GPU.
int check_gemm_common(const void* A, const void* sA, const void* B, const void* sB, int b_scale_kind, void* C,
                      int out_dtype, int accumulate, int64_t rows, int64_t N, int64_t K);

// Byte range of a workspace of `workspace_bytes` that must be zero when a
// launch starts (the arrival counters of the plan that workspace allows);
// *bytes = 0 when that plan does not split.
void gemm_workspace_zero_range(int mode, int64_t rows, int64_t N, int64_t K, int64_t groups, int num_sms,
                               size_t workspace_bytes, size_t* offset, size_t* bytes);

// Enqueue the GEMM. `status` is a device word that receives timeout codes.
// Returns cudaSuccess or the first CUDA error; *detail gets a static message.
cudaError_t launch_gemm(const GemmProblem& p, uint32_t* status, uint64_t wait_limit_ns, int debug_skip_fill,
                        int num_sms, cudaStream_t stream, const char** detail);

// The CTA-pair GEMM (gemm_pair.cu): when switched on, taken for dense
// problems large enough to fill the GPU with 256 x 256 tiles
// (pair_gemm_eligible); launch_gemm dispatches to it.
bool pair_gemm_eligible(const GemmProblem& p, int num_sms);
void set_pair_gemm_enabled(bool on);
// K split of decode-sized dense GEMMs: 0 automatic, 1 Stream-K only, 2 the
// cluster split wherever it applies.
void set_split_policy(int policy);
cudaError_t launch_gemm_pair(const GemmProblem& p, uint32_t* status, uint64_t wait_limit_ns, int debug_skip_fill,
                             cudaStream_t stream, const char** detail);

// The block-scaled GEMM (gemm_bs.cu): power-of-two row scales on both
// operands applied inside the tensor core, dense layout, FP32 output.
bool bs_gemm_eligible(const GemmProblem& p);
cudaError_t launch_gemm_bs(const GemmProblem& p, uint32_t* status, uint64_t wait_limit_ns, int debug_skip_fill,
                           int num_sms, cudaStream_t stream, const char** detail);

// Tensor-core accumulation study (see study.cu): D[128][N] = A[128][K] B[N][K]^T
// on unscaled E4M3 codes, the MMA accumulator restarted every `interval` K.
cudaError_t launch_mma_accum_study(const uint8_t* A, const uint8_t* B, float* D, int64_t N, int64_t K,
                                   int64_t interval, uint32_t* status, uint64_t wait_limit_ns, cudaStream_t stream,
                                   const char** detail);

}  // namespace fp8fg
