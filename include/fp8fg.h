/*
 * fp8fg.h -- C ABI of the fine-grained FP8 GEMM library for B300 (sm_103a).
 *
 * The method (DeepSeek-V3 report excerpt, pages 1-2; DeepGEMM article,
 * page 4):
 *   - activations are quantized to E4M3 per 1x128 tile: one FP32 scale per
 *     row (token) per 128 columns (channels);
 *   - weights are quantized to E4M3 per 128x128 block;
 *   - for the backward pass, cached FP8 activations are retiled from 1x128
 *     to 128x1 tiles (one scale per channel per 128 tokens), optionally with
 *     power-of-2 scales;
 *   - the FP8 GEMMs multiply E4M3 operands, apply both operands' scales once
 *     per 128-wide K block while promoting the partial sums to FP32, and emit
 *     BF16 or FP32; they come in a dense layout and two MoE layouts
 *     (grouped-contiguous and grouped-masked).
 *
 * Conventions shared by every entry point
 *   - Every pointer is a DEVICE pointer owned by the caller; the library
 *     never allocates or frees caller-visible memory and keeps no pointer
 *     after the call returns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). Argument checks run on the host before anything is
 *     enqueued; a non-zero return means nothing was enqueued.
 *   - Return codes: FP8FG_OK, or a negative FP8FG_ERR_* value;
 *     fp8fg_last_error_string() describes the last error of the calling
 *     thread.
 *   - Bounded device waits: a GEMM or quantizer whose internal pipeline wait
 *     runs past its limit records FP8FG_ERR_TIMEOUT in a device status word
 *     and exits; fp8fg_check() synchronizes `stream` and reports it.
 *   - Layouts are row-major. "ld(R)" below is fp8fg_scale_ld(R) = R rounded
 *     up to a multiple of 4: the row stride, in floats, of every per-row
 *     scale array, so that each row of scales starts on a 16-byte boundary
 *     (the tensor-memory-accelerator copies need it). Scale entries at
 *     positions >= R inside a padded row are neither read nor written.
 *   - E4M3 encoding: round to nearest, ties to even, saturating to +-448;
 *     the sign of zero is kept.
 *   - Scales: s = fl32(amax / 448.0f) (IEEE FP32 division), 1.0 when that
 *     is zero; with pow2 != 0, s is raised to the next power of two (kept if
 *     it already is one). Quantized value q = E4M3(fl32(x / s)).
 */
#ifndef FP8FG_H
#define FP8FG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FP8FG_API __attribute__((visibility("default")))
#else
#define FP8FG_API
#endif

typedef struct CUstream_st* fp8fg_stream_t; /* identical to cudaStream_t */

/* return codes */
#define FP8FG_OK                     0
#define FP8FG_ERR_INVALID_ARG       -1 /* null pointer, negative size, bad enum */
#define FP8FG_ERR_UNSUPPORTED_SHAPE -2 /* K, T or C not a multiple of 128; N not a multiple of 8 ... */
#define FP8FG_ERR_MISALIGNED        -3 /* a pointer is not 16-byte aligned */
#define FP8FG_ERR_CUDA              -4 /* a CUDA runtime or driver call failed */
#define FP8FG_ERR_TIMEOUT           -5 /* a bounded device wait expired */

/* element types */
#define FP8FG_BF16 0
#define FP8FG_FP32 1
#define FP8FG_E4M3 2

/* how the B operand of a GEMM is scaled */
#define FP8FG_SCALE_BLOCK128 0 /* sB[ceil(N/128)][K/128]: one scale per 128x128 block   */
#define FP8FG_SCALE_ROW      1 /* sB[K/128][ld(N)]: one scale per row per 128 K (128x1) */
#define FP8FG_SCALE_ROW_POW2 2 /* as FP8FG_SCALE_ROW, and every scale of A and of B is a power of
                                * two (fp8_requant_128x1 with pow2 = 1): dense FP32-output GEMMs
                                * then apply the scales inside the tensor core (block-scaled MMA,
                                * UE8M0) instead of promoting partial sums; other forms use the
                                * FP8FG_SCALE_ROW path. A scale that is not a power of two makes
                                * fp8fg_check report FP8FG_ERR_INVALID_ARG. */

/* what masked_m limits in fp8_gemm_grouped_masked */
#define FP8FG_MASK_ROWS 0 /* rows of A (forward / decode MoE)            */
#define FP8FG_MASK_K    1 /* the reduction extent (MoE weight gradient)  */

/* Row stride, in floats, of per-row scale arrays: rows rounded up to 4. */
FP8FG_API int64_t fp8fg_scale_ld(int64_t rows);

/*
 * fp8_quant_1x128 -- activation quantization, one scale per 1x128 tile.
 * (DeepSeek-V3 report excerpt, page 1, paragraphs 1-3: fine-grained 1x128
 * activation tiles; page 2, paragraph 1: optional power-of-2 scales.)
 *
 *   x      [M][ldx] of x_dtype (FP8FG_BF16 or FP8FG_FP32); columns [0, K) read
 *   q      [M][K]  E4M3 bytes, written
 *   s      [K/128][ld(M)] float, written: s[kb][m] scales x[m][kb*128 .. +128)
 *   pow2   0: s = amax/448; 1: power-of-2 scale
 * Requires K % 128 == 0, ldx >= K, x, q 16-byte aligned, ldx*elem % 16 == 0.
 * M == 0 or K == 0 is a no-op.
 */
FP8FG_API int fp8_quant_1x128(const void* x, int x_dtype, int64_t M, int64_t K, int64_t ldx,
                    uint8_t* q, float* s, int pow2, fp8fg_stream_t stream);

/*
 * fp8_quant_128x128 -- weight quantization, one scale per 128x128 block.
 * (Block size: the DeepSeek-V3 report's weight tiling; the pages print only
 * the activation tiles, page 1 paragraph 3.)
 *
 *   w      [G][N][K] of w_dtype (BF16 or FP32), contiguous
 *   q      [G][N][K] E4M3, written
 *   s      [G][ceil(N/128)][K/128] float, written; the last row block of a
 *          group may be partial (N % 128 rows): its amax covers those rows.
 * Requires K % 128 == 0, w and q 16-byte aligned.
 */
FP8FG_API int fp8_quant_128x128(const void* w, int w_dtype, int64_t G, int64_t N, int64_t K,
                      uint8_t* q, float* s, int pow2, fp8fg_stream_t stream);

/*
 * fp8_requant_128x1 -- backward retile from 1x128 to 128x1 tiles, written
 * transposed (channel-major, tokens contiguous) so that the weight-gradient
 * GEMM reduces over tokens along its K dimension. (DeepSeek-V3 report
 * excerpt, page 1, paragraph 3: 1x128 -> 128x1 conversion in the backward
 * pass; page 2, paragraph 1: power-of-2 scales for the activation gradient;
 * page 2, paragraph 3: the transposed-GEMM request this layout answers.)
 *
 *   src        [G][T][C]: E4M3 bytes (src_dtype FP8FG_E4M3, dequantized as
 *              fl32(decode(q) * s_src)) or BF16 / FP32 values
 *   s_src      [G][C/128][ld(T)] float, 1x128 scales of an E4M3 source
 *              (ignored otherwise, may be NULL)
 *   valid_rows NULL, or device int32 [G]: rows t >= valid_rows[g] are
 *              treated as zero (masked / padded tokens)
 *   qT         [G][C][T] E4M3, written
 *   sT         [G][T/128][ld(C)] float, written: sT[tb][c] scales tokens
 *              [tb*128, tb*128+128) of channel c
 * Requires T % 128 == 0, C % 128 == 0, 16-byte aligned src, qT and s_src.
 */
FP8FG_API int fp8_requant_128x1(const void* src, int src_dtype, const float* s_src,
                      int64_t G, int64_t T, int64_t C, const int32_t* valid_rows,
                      uint8_t* qT, float* sT, int pow2, fp8fg_stream_t stream);

/*
 * fp8_gemm_dense -- C[M][N] = sum_k Ahat[m][k] * Bhat[n][k] (C = A B^T)
 * with Ahat = q_A * sA (1x128) and Bhat = q_B * sB (128x128 blocks or
 * 128x1 rows). Partial sums of each 128-wide K block are scaled and
 * accumulated in FP32 (DeepSeek-V3 report excerpt, page 1, paragraph 3:
 * promotion to FP32 registers; outputs BF16 or FP32).
 *
 *   A          [M][K] E4M3, sA [K/128][ld(M)]
 *   B          [N][K] E4M3, sB per b_scale_kind (FP8FG_SCALE_BLOCK128 or _ROW)
 *   C          [M][N] of out_dtype (BF16 or FP32), written
 *   accumulate 1: C += result (FP32 output only: weight-gradient
 *              accumulation); 0: C = result
 *   workspace  device scratch for one of the two ways of splitting K when
 *              the output has too few tiles to occupy the GPU (at most half
 *              as many 128x128 tiles as SMs: decode-sized M). The default
 *              split runs each tile on the CTAs of a thread-block cluster,
 *              which sum their partials through distributed shared memory
 *              and need no workspace; Stream-K (chosen where the cluster
 *              split does not apply, or by fp8fg_debug_set key 4) sums them
 *              in the workspace. fp8fg_gemm_workspace_size(M, N, K) bytes,
 *              16-byte aligned, zero-filled before its first use; every call
 *              leaves its counters zero-filled again (re-zero the workspace
 *              after a call that reported FP8FG_ERR_TIMEOUT). Calls that
 *              share a workspace must not overlap on the GPU. NULL, or fewer
 *              bytes than that size, runs without Stream-K. Split tiles are
 *              summed in a fixed order: results are deterministic for a
 *              given shape, SM count and split policy, and differ from the
 *              unsplit run by FP32 rounding only.
 * Requires K % 128 == 0, N % 8 == 0, 16-byte aligned A, B, C.
 */
FP8FG_API int fp8_gemm_dense(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                   int b_scale_kind, void* C, int out_dtype, int accumulate,
                   int64_t M, int64_t N, int64_t K,
                   void* workspace, size_t workspace_bytes, fp8fg_stream_t stream);

/*
 * fp8_gemm_dense_quant -- fp8_gemm_dense with the FP8 cast of its output
 * fused in: the result, rounded to BF16, is quantized per 1x128 tile for the
 * next layer's GEMM in the GEMM's own epilogue, instead of being written in
 * BF16 and read back by fp8_quant_1x128. (DeepSeek-V3 report excerpt,
 * page 1, paragraph 3: activations quantized per 1x128 tile; page 2, last
 * paragraph: the request to fuse the FP8 cast with the data movement.)
 * Bit-identical to fp8_gemm_dense (BF16 out) followed by fp8_quant_1x128 of
 * its output.
 *
 *   A, sA, B, sB  as fp8_gemm_dense, b_scale_kind FP8FG_SCALE_BLOCK128
 *   q          [M][N] E4M3 codes of the BF16 result, written
 *   s          [N/128][ld(M)] float scales, written (the sA layout the next
 *              GEMM takes)
 *   C          NULL, or [M][N] BF16: the unquantized result as well
 *   pow2       0: s = amax/448; 1: power-of-2 scales
 *   workspace  as fp8_gemm_dense (fp8fg_gemm_workspace_size covers both)
 * Requires K % 128 == 0, N % 128 == 0, 16-byte aligned A, B, q, s (and C).
 */
FP8FG_API int fp8_gemm_dense_quant(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                   int b_scale_kind, uint8_t* q, float* s, void* C, int pow2,
                                   int64_t M, int64_t N, int64_t K,
                                   void* workspace, size_t workspace_bytes, fp8fg_stream_t stream);

/*
 * fp8_gemm_dgrad -- data gradient of a Linear layer whose forward pass is
 * Y[M][N] = X[M][K] W[N][K]^T:  dX[M][K] = dY[M][N] W[N][K], all in FP8
 * (DeepSeek-V3 report excerpt, page 1, paragraph 3: Fprop, Dgrad and Wgrad
 * run as FP8 GEMMs; page 2, paragraph 3: the request for transposed-GEMM
 * support). W is read as its own transpose straight from the forward
 * pass's E4M3 bytes and 128x128 block scales (a block's scale does not
 * change under transposition); no transposed copy is made.
 *
 *   dY    [M][N] E4M3, s_dY [N/128][ld(M)]: dY quantized per 1x128 tile
 *         along N (fp8_quant_1x128)
 *   W     [N][K] E4M3, sW [N/128][K/128]: as fp8_quant_128x128 wrote them
 *   dX    [M][K] of out_dtype (BF16 or FP32), written (accumulate = 1:
 *         dX += result, FP32 only)
 *   workspace  as fp8_gemm_dense with (M, K, N): fp8fg_gemm_workspace_size(M, K, N)
 * Requires N % 128 == 0, K % 16 == 0, 16-byte aligned dY, W, dX, s_dY.
 */
FP8FG_API int fp8_gemm_dgrad(const uint8_t* dY, const float* s_dY, const uint8_t* W, const float* sW, void* dX,
                             int out_dtype, int accumulate, int64_t M, int64_t N, int64_t K,
                             void* workspace, size_t workspace_bytes, fp8fg_stream_t stream);

/*
 * fp8_gemm_dense_noalloc -- fp8_gemm_dense for callers that cannot allocate
 * device memory. (No counterpart in the paper: a deployment convenience of
 * this library.) Some callers only receive device pointers from a host
 * application that owns all device memory and offers no allocator, or run
 * where a device allocation is forbidden (it can synchronize the device);
 * they cannot provide the Stream-K workspace. This entry point computes the
 * same product with the same arguments minus the workspace, using instead a
 * 64 MiB array that is part of the library's device code. It allocates
 * nothing.
 *   - The CUDA runtime loads device code lazily by default, so the array is
 *     committed on a device by the first call there (which also looks up its
 *     address). That first call may fail for lack of device memory or
 *     synchronize the device: make it at start-up, outside latency-critical
 *     code and before any stream capture. The array is then held on that
 *     device until the process exits.
 *   - All calls share the array: calls whose GPU work overlaps race on it.
 *   - Each call clears the part of the array that must start at zero.
 *   - Arguments are checked as fp8_gemm_dense checks them; a shape needing
 *     more scratch than 64 MiB is rejected with FP8FG_ERR_UNSUPPORTED_SHAPE
 *     (none exists on GPUs with up to ~170 SMs).
 */
FP8FG_API int fp8_gemm_dense_noalloc(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                     int b_scale_kind, void* C, int out_dtype, int accumulate,
                                     int64_t M, int64_t N, int64_t K, fp8fg_stream_t stream);

/* Bytes of workspace fp8_gemm_dense and fp8_gemm_dense_quant use for this
 * shape on the current device (0 if neither splits tiles along K); one
 * workspace of this size serves both. Needs a CUDA device; 0 on error. */
FP8FG_API size_t fp8fg_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * fp8_gemm_grouped_contig -- MoE GEMM, grouped-contiguous layout (DeepGEMM
 * article, page 4: "dense and two MoE layouts").
 * Token rows of A are sorted by expert; each expert's segment is padded to
 * a multiple of 128 rows; m_indices[row] is the row's expert id, or -1 for a
 * padding row. Row r of C is A[r] * B[m_indices[r]]^T; padding rows of C are
 * not written.
 *
 *   A          [M_total][K] E4M3, sA [K/128][ld(M_total)]
 *   B          [E][N][K] E4M3,    sB [E][ceil(N/128)][K/128]
 *   m_indices  device int32 [M_total], values in [-1, E)
 *   C          [M_total][N] of out_dtype
 * Requires M_total % 128 == 0, K % 128 == 0, N % 8 == 0; every aligned
 * 128-row block holds one expert (or only padding).
 */
FP8FG_API int fp8_gemm_grouped_contig(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                            const int32_t* m_indices, void* C, int out_dtype,
                            int64_t M_total, int64_t N, int64_t K, int64_t E,
                            fp8fg_stream_t stream);

/*
 * fp8_gemm_grouped_masked -- MoE GEMM, grouped-masked layout (DeepGEMM
 * article, page 4; decode batches of at most 256 tokens per expert,
 * DeepSeek-V3 report excerpt, page 2, paragraph 3).
 *
 * mask_dim FP8FG_MASK_ROWS (forward/decode): for each expert e, rows
 *   [0, masked_m[e]) of C[e] = A[e] B[e]^T; rows >= masked_m[e] of C[e] are
 *   not written.
 *   A [E][M_max][K], sA [E][K/128][ld(M_max)]; B [E][N][K];
 *   sB [E][ceil(N/128)][K/128] (BLOCK128) or [E][K/128][ld(N)] (ROW);
 *   C [E][M_max][N].
 * mask_dim FP8FG_MASK_K (MoE weight gradient, dW_e = G_e^T X_e over the
 *   expert's tokens): the reduction of expert e runs over K positions
 *   [0, roundup(masked_m[e], 128)); A = G_e^T [E][M_max][K] with
 *   sA [E][K/128][ld(M_max)], B = X_e^T [E][N][K] with b_scale_kind ROW
 *   sB [E][K/128][ld(N)]; every row of C[e] is written (zero for an
 *   expert without tokens, unchanged when accumulate is 1).
 *
 *   masked_m   device int32 [E], values in [0, M_max] (ROWS) or [0, K] (K)
 *   expected_m host hint of the typical masked_m, >= 0. Reserved: checked
 *              but not used by this version (the kernel finds the active
 *              tiles from masked_m on the device, whatever the counts)
 *   accumulate FP32 output only, as in fp8_gemm_dense
 * Requires K % 128 == 0, N % 8 == 0, 16-byte aligned A, B, C.
 */
FP8FG_API int fp8_gemm_grouped_masked(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                            int b_scale_kind, const int32_t* masked_m, int mask_dim,
                            void* C, int out_dtype, int accumulate,
                            int64_t E, int64_t M_max, int64_t N, int64_t K, int64_t expected_m,
                            fp8fg_stream_t stream);

/*
 * fp8fg_check -- synchronize `stream`, then report a device-side error
 * recorded by an earlier call on this device (FP8FG_ERR_TIMEOUT) or a
 * CUDA error (FP8FG_ERR_CUDA), and clear the recorded status.
 */
FP8FG_API int fp8fg_check(fp8fg_stream_t stream);

/* Description of the calling thread's last error ("" if none). */
FP8FG_API const char* fp8fg_last_error_string(void);

/* Library version string. */
FP8FG_API const char* fp8fg_version(void);

/*
 * fp8fg_study_mma_accumulation -- measurement of the tensor core's own FP8
 * accumulation (no counterpart on the GEMM path; the DeepSeek-V3 report
 * excerpt, page 1 paragraph 1 and page 2 paragraph 1, measured the H800's:
 * about 14 bits kept, ~2% error at K=4096 without promotion).
 *
 *   A        [128][K] E4M3 codes, used unscaled (scale 1)
 *   B        [N][K]   E4M3 codes, unscaled
 *   D        [128][N] float, written: sum over k of A[m][k] * B[n][k], where
 *            the tensor-core accumulator restarts every `interval` K
 *            elements and each restarted partial is added into FP32 (IEEE
 *            round-to-nearest add). interval >= K: one chained accumulator
 *            (no promotion); 128: the GEMM path's promotion interval.
 * Requires K % 128 == 0, N % 128 == 0, interval % 32 == 0 (> 0), 16-byte
 * aligned pointers. Slow by design (one CTA per 128 columns, serial).
 */
FP8FG_API int fp8fg_study_mma_accumulation(const uint8_t* A, const uint8_t* B, float* D, int64_t N, int64_t K,
                                           int64_t interval, fp8fg_stream_t stream);

/*
 * fp8fg_debug_set -- test hooks (no counterpart in the method):
 *   key 1: wait limit of the bounded device waits, in nanoseconds (value 0
 *          restores the default of 2 s);
 *   key 2: the TMA producer of every GEMM and quantizer CTA skips the copy
 *          of its k-th pipeline fill (value k >= 0; -1 disables), so that
 *          the consumers' bounded waits run out and the call reports
 *          FP8FG_ERR_TIMEOUT without faulting;
 *   key 3: 1 sends large dense GEMMs (more 128x256 tiles than half the
 *          SMs) to the CTA-pair kernel (tcgen05 cta_group::2, 256 x 256
 *          tiles); 0 (the default) keeps every GEMM on the single-CTA
 *          kernel. The environment variable FP8FG_PAIR=1 sets 1 at load.
 *   key 4: how decode-sized dense GEMMs (128 x 128 output tiles at most
 *          half the SMs) split K: 0 (the default) automatic, 1 Stream-K
 *          over the caller's workspace only, 2 the cluster split (the CTAs
 *          of a thread-block cluster share a tile and sum their partials
 *          through distributed shared memory; no workspace) wherever it
 *          applies. FP8FG_SPLIT=stream|cluster sets 1 or 2 at load.
 * Returns FP8FG_OK or FP8FG_ERR_INVALID_ARG.
 */
FP8FG_API int fp8fg_debug_set(int key, int64_t value);

/*
 * Environment variables, read once per process when first needed (tuning
 * and A/B switches; results stay within the same tolerances):
 *   FP8FG_BN=128|192|256   tile width of every single-CTA GEMM (default:
 *                          128 for dense problems of one 128-row block,
 *                          else 256; MN-major B takes 256 for 192);
 *   FP8FG_SPLIT=stream|cluster  K split of decode-sized dense GEMMs (key 4);
 *   FP8FG_PAIR=1           large dense GEMMs on the CTA-pair kernel (key 3);
 *   FP8FG_ISSUERS=1        one MMA-issuing warp instead of two;
 *   FP8FG_PDL=0            no programmatic dependent launch.
 */

#ifdef __cplusplus
}
#endif

#endif /* FP8FG_H */
