// C ABI of the library: argument checks, per-device state and error
// reporting around the launchers in quant.cu and gemm.cu. The declarations
// and the contract of every entry point are in include/fp8fg.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/fp8fg.h"
#include "common.cuh"
#include "kernels.h"

namespace {

// Device-side status word written by bounded waits that give up. A file-scope
// device variable: no allocation; its device address is looked up per device.
__device__ uint32_t g_status_word[1];

thread_local std::string t_last_error;

constexpr uint64_t kDefaultWaitNs = 2ull * 1000 * 1000 * 1000;
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};
std::atomic<int> g_debug_skip_fill{-1};

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  uint32_t* status = nullptr;
};
DeviceState g_dev[64];
std::mutex g_dev_mu;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(FP8FG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Per-device state for the current device; nullptr (with the error set) on failure.
const DeviceState* device_state(int* err) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *err = cuda_fail(e == cudaSuccess ? cudaErrorInvalidDevice : e, "cudaGetDevice");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      *err = cuda_fail(e, "cudaDeviceGetAttribute(multiProcessorCount)");
      return nullptr;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) {
      *err = cuda_fail(e, "cudaGetSymbolAddress(status word)");
      return nullptr;
    }
    st.status = static_cast<uint32_t*>(p);
    st.ready = true;
  }
  return &st;
}

fp8fg::QuantLaunch quant_launch(const DeviceState* st) {
  return fp8fg::QuantLaunch{st->num_sms, st->status, g_wait_limit_ns.load(), g_debug_skip_fill.load()};
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int64_t elem_size(int dtype) {
  switch (dtype) {
    case FP8FG_BF16: return 2;
    case FP8FG_FP32: return 4;
    case FP8FG_E4M3: return 1;
    default: return 0;
  }
}

constexpr int64_t kMaxDim = (1ll << 31) - 1;

}  // namespace

namespace fp8fg {
int check_gemm_common(const void* A, const void* sA, const void* B, const void* sB, int b_scale_kind, void* C,
                      int out_dtype, int accumulate, int64_t rows, int64_t N, int64_t K) {
  if (rows < 0 || N < 0 || K < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
  if (out_dtype != FP8FG_BF16 && out_dtype != FP8FG_FP32)
    return fail(FP8FG_ERR_INVALID_ARG, "out_dtype must be FP8FG_BF16 or FP8FG_FP32");
  if (b_scale_kind != FP8FG_SCALE_BLOCK128 && b_scale_kind != FP8FG_SCALE_ROW && b_scale_kind != FP8FG_SCALE_ROW_POW2)
    return fail(FP8FG_ERR_INVALID_ARG,
                "b_scale_kind must be FP8FG_SCALE_BLOCK128, FP8FG_SCALE_ROW or FP8FG_SCALE_ROW_POW2");
  if (accumulate != 0 && accumulate != 1) return fail(FP8FG_ERR_INVALID_ARG, "accumulate must be 0 or 1");
  if (accumulate && out_dtype != FP8FG_FP32)
    return fail(FP8FG_ERR_INVALID_ARG, "accumulate=1 needs FP32 output");
  if (K == 0 || K % 128 != 0) return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a positive multiple of 128", (long long)K);
  if (N % 8 != 0) return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "N=%lld must be a multiple of 8", (long long)N);
  if (rows > kMaxDim || N > kMaxDim || K > kMaxDim) return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "dimension too large");
  if (!A || !sA || !B || !sB || !C) return fail(FP8FG_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(sA))
    return fail(FP8FG_ERR_MISALIGNED, "A, B, C and sA must be 16-byte aligned");
  if (b_scale_kind != FP8FG_SCALE_BLOCK128 ? !aligned16(sB) : !aligned4(sB))
    return fail(FP8FG_ERR_MISALIGNED, "sB must be 16-byte aligned (per-row scales) or 4-byte aligned");
  return FP8FG_OK;
}
}  // namespace fp8fg

namespace {
using fp8fg::check_gemm_common;

int run_gemm(const fp8fg::GemmProblem& p, cudaStream_t stream) {
  int err = FP8FG_OK;
  const DeviceState* st = device_state(&err);
  if (!st) return err;
  const char* detail = "";
  cudaError_t e = fp8fg::launch_gemm(p, st->status, g_wait_limit_ns.load(), g_debug_skip_fill.load(), st->num_sms,
                                     stream, &detail);
  if (e != cudaSuccess) return cuda_fail(e, detail);
  return FP8FG_OK;
}

}  // namespace

namespace fp8fg {
void set_last_error(const char* msg) { t_last_error = msg; }
}  // namespace fp8fg

extern "C" {

int64_t fp8fg_scale_ld(int64_t rows) { return rows <= 0 ? 0 : (rows + 3) / 4 * 4; }

const char* fp8fg_version(void) { return "fp8fg 0.1.0 (sm_103a)"; }

const char* fp8fg_last_error_string(void) { return t_last_error.c_str(); }

int fp8_quant_1x128(const void* x, int x_dtype, int64_t M, int64_t K, int64_t ldx, uint8_t* q, float* s, int pow2,
                    fp8fg_stream_t stream) {
  if (M < 0 || K < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
  if (x_dtype != FP8FG_BF16 && x_dtype != FP8FG_FP32)
    return fail(FP8FG_ERR_INVALID_ARG, "x_dtype must be FP8FG_BF16 or FP8FG_FP32");
  if (pow2 != 0 && pow2 != 1) return fail(FP8FG_ERR_INVALID_ARG, "pow2 must be 0 or 1");
  if (K % 128 != 0) return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a multiple of 128", (long long)K);
  if (M == 0 || K == 0) return FP8FG_OK;
  if (ldx < K) return fail(FP8FG_ERR_INVALID_ARG, "ldx < K");
  if (!x || !q || !s) return fail(FP8FG_ERR_INVALID_ARG, "null pointer");
  const int64_t esz = elem_size(x_dtype);
  if (!aligned16(x) || !aligned16(q) || !aligned16(s) || (ldx * esz) % 16 != 0)
    return fail(FP8FG_ERR_MISALIGNED, "x, q, s must be 16-byte aligned and ldx*elem a multiple of 16 bytes");
  int err = FP8FG_OK;
  const DeviceState* st = device_state(&err);
  if (!st) return err;
  cudaError_t e = fp8fg::launch_quant_1x128(x, x_dtype == FP8FG_FP32, M, K, ldx, q, s, fp8fg_scale_ld(M), pow2,
                                            quant_launch(st), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8FG_OK : cuda_fail(e, "quant_1x128 launch");
}

int fp8_quant_128x128(const void* w, int w_dtype, int64_t G, int64_t N, int64_t K, uint8_t* q, float* s, int pow2,
                      fp8fg_stream_t stream) {
  if (G < 0 || N < 0 || K < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
  if (w_dtype != FP8FG_BF16 && w_dtype != FP8FG_FP32)
    return fail(FP8FG_ERR_INVALID_ARG, "w_dtype must be FP8FG_BF16 or FP8FG_FP32");
  if (pow2 != 0 && pow2 != 1) return fail(FP8FG_ERR_INVALID_ARG, "pow2 must be 0 or 1");
  if (K % 128 != 0) return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a multiple of 128", (long long)K);
  if (G == 0 || N == 0 || K == 0) return FP8FG_OK;
  if (!w || !q || !s) return fail(FP8FG_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(w) || !aligned16(q) || !aligned4(s))
    return fail(FP8FG_ERR_MISALIGNED, "w, q must be 16-byte aligned, s 4-byte aligned");
  int err = FP8FG_OK;
  const DeviceState* st = device_state(&err);
  if (!st) return err;
  cudaError_t e = fp8fg::launch_quant_128x128(w, w_dtype == FP8FG_FP32, G, N, K, q, s, pow2, quant_launch(st),
                                              reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8FG_OK : cuda_fail(e, "quant_128x128 launch");
}

int fp8_requant_128x1(const void* src, int src_dtype, const float* s_src, int64_t G, int64_t T, int64_t C,
                      const int32_t* valid_rows, uint8_t* qT, float* sT, int pow2, fp8fg_stream_t stream) {
  if (G < 0 || T < 0 || C < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
  if (src_dtype != FP8FG_E4M3 && src_dtype != FP8FG_BF16 && src_dtype != FP8FG_FP32)
    return fail(FP8FG_ERR_INVALID_ARG, "src_dtype must be FP8FG_E4M3, FP8FG_BF16 or FP8FG_FP32");
  if (pow2 != 0 && pow2 != 1) return fail(FP8FG_ERR_INVALID_ARG, "pow2 must be 0 or 1");
  if (T % 128 != 0 || C % 128 != 0)
    return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "T=%lld and C=%lld must be multiples of 128", (long long)T, (long long)C);
  if (G == 0 || T == 0 || C == 0) return FP8FG_OK;
  if (!src || !qT || !sT || (src_dtype == FP8FG_E4M3 && !s_src)) return fail(FP8FG_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(src) || !aligned16(qT) || !aligned4(sT) || (s_src && !aligned16(s_src)))
    return fail(FP8FG_ERR_MISALIGNED, "src, qT and s_src must be 16-byte aligned, sT 4-byte aligned");
  if (valid_rows && !aligned4(valid_rows)) return fail(FP8FG_ERR_MISALIGNED, "valid_rows must be 4-byte aligned");
  int err = FP8FG_OK;
  const DeviceState* st = device_state(&err);
  if (!st) return err;
  const int kind = src_dtype == FP8FG_E4M3 ? 0 : (src_dtype == FP8FG_BF16 ? 1 : 2);
  cudaError_t e = fp8fg::launch_requant_128x1(src, kind, s_src, fp8fg_scale_ld(T), G, T, C, valid_rows, qT, sT,
                                              fp8fg_scale_ld(C), pow2, quant_launch(st),
                                              reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8FG_OK : cuda_fail(e, "requant_128x1 launch");
}

size_t fp8fg_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 128 != 0) return 0;
  int err = FP8FG_OK;
  const DeviceState* st = device_state(&err);
  if (!st) return 0;
  return fp8fg::gemm_workspace_bytes(fp8fg::kModeDense, M, N, K, 1, st->num_sms);
}

int fp8_gemm_dense(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, int b_scale_kind, void* C,
                   int out_dtype, int accumulate, int64_t M, int64_t N, int64_t K, void* workspace,
                   size_t workspace_bytes, fp8fg_stream_t stream) {
  if (M == 0 || N == 0) {
    if (M < 0 || N < 0 || K < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
    return FP8FG_OK;
  }
  int rc = check_gemm_common(A, sA, B, sB, b_scale_kind, C, out_dtype, accumulate, M, N, K);
  if (rc) return rc;
  fp8fg::GemmProblem p{};
  p.mode = fp8fg::kModeDense;
  p.A = A; p.sA = sA; p.B = B; p.sB = sB;
  p.b_row = b_scale_kind != FP8FG_SCALE_BLOCK128;
  p.b_scale_pow2 = b_scale_kind == FP8FG_SCALE_ROW_POW2;
  p.C = C; p.out_f32 = out_dtype == FP8FG_FP32; p.accumulate = accumulate;
  p.rows = M; p.N = N; p.K = K; p.groups = 1; p.groupsB = 1;
  if (workspace != nullptr && !aligned16(workspace))
    return fail(FP8FG_ERR_MISALIGNED, "workspace must be 16-byte aligned");
  p.workspace = workspace;
  p.workspace_bytes = workspace ? workspace_bytes : 0;
  return run_gemm(p, reinterpret_cast<cudaStream_t>(stream));
}

int fp8_gemm_dense_quant(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, int b_scale_kind,
                         uint8_t* q, float* s, void* C, int pow2, int64_t M, int64_t N, int64_t K, void* workspace,
                         size_t workspace_bytes, fp8fg_stream_t stream) {
  if (M == 0 || N == 0) {
    if (M < 0 || N < 0 || K < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
    return FP8FG_OK;
  }
  if (pow2 != 0 && pow2 != 1) return fail(FP8FG_ERR_INVALID_ARG, "pow2 must be 0 or 1");
  if (!q || !s) return fail(FP8FG_ERR_INVALID_ARG, "null pointer");
  // the common checks, with q standing in for C when no BF16 C is wanted
  int rc = check_gemm_common(A, sA, B, sB, b_scale_kind, C ? C : static_cast<void*>(q), FP8FG_BF16, 0, M, N, K);
  if (rc) return rc;
  if (b_scale_kind != FP8FG_SCALE_BLOCK128)
    return fail(FP8FG_ERR_INVALID_ARG, "fused quantization takes 128x128 block-scaled B");
  if (N % 128 != 0) return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "N=%lld must be a multiple of 128", (long long)N);
  if (!aligned16(q) || !aligned16(s)) return fail(FP8FG_ERR_MISALIGNED, "q and s must be 16-byte aligned");
  fp8fg::GemmProblem p{};
  p.mode = fp8fg::kModeDense;
  p.A = A; p.sA = sA; p.B = B; p.sB = sB; p.b_row = 0;
  p.C = C; p.out_f32 = 0; p.accumulate = 0;
  p.rows = M; p.N = N; p.K = K; p.groups = 1; p.groupsB = 1;
  p.q_out = q; p.s_out = s; p.pow2_out = pow2;
  if (workspace != nullptr && !aligned16(workspace))
    return fail(FP8FG_ERR_MISALIGNED, "workspace must be 16-byte aligned");
  p.workspace = workspace;
  p.workspace_bytes = workspace ? workspace_bytes : 0;
  return run_gemm(p, reinterpret_cast<cudaStream_t>(stream));
}

int fp8_gemm_dgrad(const uint8_t* dY, const float* s_dY, const uint8_t* W, const float* sW, void* dX, int out_dtype,
                   int accumulate, int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                   fp8fg_stream_t stream) {
  if (M == 0 || K == 0) {
    if (M < 0 || N < 0 || K < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
    return FP8FG_OK;
  }
  // as a GEMM: rows M, output columns K, reduction N; B = W read MN-major
  int rc = check_gemm_common(dY, s_dY, W, sW, FP8FG_SCALE_BLOCK128, dX, out_dtype, accumulate, M, K, N);
  if (rc) return rc;
  if (K % 16 != 0) return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a multiple of 16", (long long)K);
  fp8fg::GemmProblem p{};
  p.mode = fp8fg::kModeDense;
  p.A = dY; p.sA = s_dY; p.B = W; p.sB = sW; p.b_row = 0; p.b_mn_major = 1;
  p.C = dX; p.out_f32 = out_dtype == FP8FG_FP32; p.accumulate = accumulate;
  p.rows = M; p.N = K; p.K = N; p.groups = 1; p.groupsB = 1;
  if (workspace != nullptr && !aligned16(workspace))
    return fail(FP8FG_ERR_MISALIGNED, "workspace must be 16-byte aligned");
  p.workspace = workspace;
  p.workspace_bytes = workspace ? workspace_bytes : 0;
  return run_gemm(p, reinterpret_cast<cudaStream_t>(stream));
}

int fp8_gemm_grouped_contig(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                            const int32_t* m_indices, void* C, int out_dtype, int64_t M_total, int64_t N, int64_t K,
                            int64_t E, fp8fg_stream_t stream) {
  if (E < 0 || M_total < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
  if (M_total % 128 != 0)
    return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "M_total=%lld must be a multiple of 128", (long long)M_total);
  if (M_total == 0 || N == 0 || E == 0) {
    if (N < 0 || K < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
    return FP8FG_OK;
  }
  int rc = check_gemm_common(A, sA, B, sB, FP8FG_SCALE_BLOCK128, C, out_dtype, 0, M_total, N, K);
  if (rc) return rc;
  if (!m_indices || !aligned4(m_indices)) return fail(FP8FG_ERR_INVALID_ARG, "m_indices must be a 4-byte aligned device pointer");
  if (E > kMaxDim) return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "too many experts");
  fp8fg::GemmProblem p{};
  p.mode = fp8fg::kModeContig;
  p.A = A; p.sA = sA; p.B = B; p.sB = sB; p.b_row = 0;
  p.C = C; p.out_f32 = out_dtype == FP8FG_FP32; p.accumulate = 0;
  p.rows = M_total; p.N = N; p.K = K; p.groups = 1; p.groupsB = E;
  p.m_indices = m_indices;
  return run_gemm(p, reinterpret_cast<cudaStream_t>(stream));
}

int fp8_gemm_grouped_masked(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, int b_scale_kind,
                            const int32_t* masked_m, int mask_dim, void* C, int out_dtype, int accumulate, int64_t E,
                            int64_t M_max, int64_t N, int64_t K, int64_t expected_m, fp8fg_stream_t stream) {
  (void)expected_m;
  if (E < 0 || M_max < 0 || expected_m < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
  if (mask_dim != FP8FG_MASK_ROWS && mask_dim != FP8FG_MASK_K)
    return fail(FP8FG_ERR_INVALID_ARG, "mask_dim must be FP8FG_MASK_ROWS or FP8FG_MASK_K");
  if (E == 0 || M_max == 0 || N == 0) {
    if (N < 0 || K < 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size");
    return FP8FG_OK;
  }
  int rc = check_gemm_common(A, sA, B, sB, b_scale_kind, C, out_dtype, accumulate, M_max, N, K);
  if (rc) return rc;
  if (!masked_m || !aligned4(masked_m)) return fail(FP8FG_ERR_INVALID_ARG, "masked_m must be a 4-byte aligned device pointer");
  if (E > kMaxDim) return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "too many experts");
  fp8fg::GemmProblem p{};
  p.mode = mask_dim == FP8FG_MASK_ROWS ? fp8fg::kModeMaskedRows : fp8fg::kModeMaskedK;
  p.A = A; p.sA = sA; p.B = B; p.sB = sB; p.b_row = b_scale_kind != FP8FG_SCALE_BLOCK128;
  p.C = C; p.out_f32 = out_dtype == FP8FG_FP32; p.accumulate = accumulate;
  p.rows = M_max; p.N = N; p.K = K; p.groups = E; p.groupsB = E;
  p.masked = masked_m;
  return run_gemm(p, reinterpret_cast<cudaStream_t>(stream));
}

int fp8fg_check(fp8fg_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int err = FP8FG_OK;
  const DeviceState* st = device_state(&err);
  if (!st) return err;
  uint32_t word = 0;
  e = cudaMemcpy(&word, st->status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (word != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpy(st->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    if (word == fp8fg::kStatusScaleNotPow2)
      return fail(FP8FG_ERR_INVALID_ARG,
                  "a GEMM with FP8FG_SCALE_ROW_POW2 was given a scale that is not a power of two (its result is wrong)");
    return fail(FP8FG_ERR_TIMEOUT, "a bounded device wait expired (code %u)", word);
  }
  return FP8FG_OK;
}

int fp8fg_study_mma_accumulation(const uint8_t* A, const uint8_t* B, float* D, int64_t N, int64_t K,
                                 int64_t interval, fp8fg_stream_t stream) {
  if (N < 0 || K < 0 || interval <= 0) return fail(FP8FG_ERR_INVALID_ARG, "negative size or interval <= 0");
  if (K % 128 != 0 || N % 128 != 0 || interval % 32 != 0)
    return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "K and N must be multiples of 128, interval a multiple of 32");
  if (N == 0 || K == 0) return FP8FG_OK;
  if (N > kMaxDim || K > kMaxDim) return fail(FP8FG_ERR_UNSUPPORTED_SHAPE, "dimension too large");
  if (!A || !B || !D) return fail(FP8FG_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(A) || !aligned16(B) || !aligned16(D)) return fail(FP8FG_ERR_MISALIGNED, "A, B, D must be 16-byte aligned");
  int err = FP8FG_OK;
  const DeviceState* st = device_state(&err);
  if (!st) return err;
  const char* detail = "";
  cudaError_t e = fp8fg::launch_mma_accum_study(A, B, D, N, K, interval, st->status, g_wait_limit_ns.load(),
                                                reinterpret_cast<cudaStream_t>(stream), &detail);
  return e == cudaSuccess ? FP8FG_OK : cuda_fail(e, detail);
}

int fp8fg_debug_set(int key, int64_t value) {
  switch (key) {
    case 1:
      if (value < 0) return fail(FP8FG_ERR_INVALID_ARG, "wait limit must be >= 0");
      g_wait_limit_ns.store(value == 0 ? kDefaultWaitNs : static_cast<uint64_t>(value));
      return FP8FG_OK;
    case 2:
      if (value < -1 || value > 0x7FFFFFFF) return fail(FP8FG_ERR_INVALID_ARG, "bad fill index");
      g_debug_skip_fill.store(static_cast<int>(value));
      return FP8FG_OK;
    case 3:
      if (value != 0 && value != 1) return fail(FP8FG_ERR_INVALID_ARG, "value must be 0 or 1");
      fp8fg::set_pair_gemm_enabled(value == 1);
      return FP8FG_OK;
    case 4:
      if (value < 0 || value > 2) return fail(FP8FG_ERR_INVALID_ARG, "value must be 0, 1 or 2");
      fp8fg::set_split_policy(static_cast<int>(value));
      return FP8FG_OK;
    default:
      return fail(FP8FG_ERR_INVALID_ARG, "unknown debug key %d", key);
  }
}

}  // extern "C"
