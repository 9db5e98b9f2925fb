/*
 * fp8bs -- fine-grained block-scaled FP8 GEMM path for B300 (sm_103a).
 *
 * C ABI of libfp8bs.so. Plain pointers and sizes only.
 *
 * The method (fine-grained FP8 mixed precision):
 *  - activations are grouped and scaled per 1x128 tile (per token per 128
 *    channels), weights per 128x128 block (per 128 input channels per 128
 *    output channels) -- "personal notes concerning the deepseek core
 *    readings" (why-be.why-be.co.kr), fine-grained quantization paragraph,
 *    Figure 7(a);
 *  - each group's maximum magnitude is mapped onto the largest FP8 value and
 *    the tensor is quantized online with that factor -- Q&A post on
 *    xn--9g3bo1gtkw0l8ubf92bgle.kr, mixed-precision paragraph;
 *  - the GEMM multiplies the FP8 operands on tensor cores and applies the
 *    per-group scales along K on CUDA cores while promoting partial sums to
 *    FP32 -- same Q&A post, paragraph on per-group scaling factors along K,
 *    and "How Google Is Changing How We Method Deepseek", paragraph on
 *    limited accumulation bit width;
 *  - in MoE, activations are quantized before the up-projection and each
 *    expert runs an FP8 GEMM (FP8 Fprop) -- Q&A post, paragraph on
 *    quantizing before the MoE up-projections.
 *
 * Numerics fixed by the statement of the problem: FP8 = E4M3 (OCP "FN"
 * variant, max 448); group scale s = amax / 448 in binary32 (s = 1 when the
 * group is all zeros); code q = round-to-nearest-even-with-saturation of the
 * binary32 quotient x / s. The stored scale s is the dequantization
 * multiplier: value ~= decode(q) * s.
 *
 * Conventions for every call:
 *  - All tensor pointers are caller-owned DEVICE memory on the current CUDA
 *    device. The library allocates and frees nothing and never synchronizes,
 *    except fp8bs_last_device_error.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously. The GEMM calls are launched as
 *    programmatic dependents of the previous kernel on the stream: their
 *    set-up may overlap that kernel's end, but they read and write no global
 *    memory before it has completed, so stream order holds as for any launch.
 *  - Arguments are validated before anything is launched; a rejected call
 *    returns FP8BS_ERR_INVALID_ARG or FP8BS_ERR_UNSUPPORTED and touches no
 *    memory. A launch failure returns FP8BS_ERR_CUDA. Errors detected on the
 *    device (a bounded wait that expired, bad expert offsets) are reported
 *    later by fp8bs_last_device_error.
 *  - M = 0 (or an expert with no rows) is a valid no-op.
 *  - Inputs must be finite; NaN/Inf inputs are outside the contract.
 *  - Leading dimensions are in elements; rows must start on 16-byte
 *    boundaries (pointers 16-byte aligned, ld * element size % 16 == 0).
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *fp8bs_stream_t;

typedef enum {
    FP8BS_OK = 0,
    FP8BS_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative size, bad stride */
    FP8BS_ERR_UNSUPPORTED = 2, /* K or N not a multiple of 128, too many experts, wrong GPU */
    FP8BS_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    FP8BS_ERR_TIMEOUT = 4      /* a device-side bounded wait expired (see last_device_error) */
} fp8bs_status;

typedef enum { FP8BS_OUT_F32 = 0, FP8BS_OUT_BF16 = 1 } fp8bs_out_dtype;

/*
 * Output tile of the GEMM kernels (all give identical results; they differ
 * only in speed). AUTO picks, when N % 256 == 0, PAIR_256x256 for dense
 * GEMMs with M > 128 and 128x256 for grouped GEMMs; else (N % 256 != 0,
 * or a dense GEMM with M <= 128) 128x128. The PAIR shapes run a CTA pair
 * (thread-block cluster of 2) per tile with the pair-wide tensor-core MMA;
 * PAIR_256x256 needs N % 256 == 0. The PAIR shapes write bf16 output with
 * TMA stores that overlap the next tile; the others store synchronously.
 */
typedef enum {
    FP8BS_TILE_AUTO = 0,
    FP8BS_TILE_128x256 = 1,
    FP8BS_TILE_128x128 = 2,
    FP8BS_TILE_PAIR_256x256 = 3,
    FP8BS_TILE_PAIR_256x128 = 4
} fp8bs_tile;

/*
 * Activation quantization, 1x128 tiles (per token per 128 channels).
 *
 *   x      bf16  [M, K], row stride ldx (elements)            (input)
 *   q      e4m3  [M, K], row stride ldq (bytes)               (output codes)
 *   scale  fp32  [M, K/128] row-major, contiguous             (output)
 *
 * For every row m and group g: amax = max_k |x[m, 128g+k]|,
 * s = scale[m, g] = amax/448 (1 if amax == 0), q[m, 128g+k] = E4M3(x/s).
 * K % 128 == 0 (else FP8BS_ERR_UNSUPPORTED). Codes and scales are
 * bit-identical to the definition above.
 */
fp8bs_status fp8bs_quantize_act_1x128(const void *x, int64_t M, int64_t K, int64_t ldx,
                                      uint8_t *q, int64_t ldq, float *scale,
                                      fp8bs_stream_t stream);

/*
 * The two quantizers with power-of-two scales: s = 2^e for the smallest
 * integer e in [-127, 127] with amax / 2^e <= 448 (s = 1 for an all-zero
 * group), i.e. scales that the UE8M0 scale format of Blackwell's
 * microscaling MMA can hold ("How I Improved My Deepseek In In The Future"
 * points to Blackwell microscaling as the direction of FP8 hardware). Codes
 * are E4M3(x / s) as before, now with an exact division. Layouts, checks and
 * the GEMM that consumes the scales are unchanged; only the scale values
 * differ (at most 2x larger than amax / 448, so codes use [224, 448] for each
 * group's largest magnitude instead of exactly 448).
 */
fp8bs_status fp8bs_quantize_act_1x128_pow2(const void *x, int64_t M, int64_t K, int64_t ldx,
                                           uint8_t *q, int64_t ldq, float *scale,
                                           fp8bs_stream_t stream);
fp8bs_status fp8bs_quantize_weight_128x128_pow2(const void *w, int64_t N, int64_t K, int64_t ldw,
                                                uint8_t *q, int64_t ldq, float *scale,
                                                fp8bs_stream_t stream);

/*
 * Both quantizations of an FP8 linear layer in one launch: the activations
 * x [M, K] in 1x128 tiles (as fp8bs_quantize_act_1x128) and the weights
 * w [N, Kw] in 128x128 blocks (as fp8bs_quantize_weight_128x128). The two are
 * independent; one launch lets them share the GPU instead of running back to
 * back. Codes and scales are bit-identical to the two separate calls; the
 * arguments, layouts and checks are theirs. Either part may be empty
 * (M == 0 or N == 0).
 */
fp8bs_status fp8bs_quantize_act_and_weight(const void *x, int64_t M, int64_t K, int64_t ldx,
                                           uint8_t *qx, int64_t ldqx, float *sx, const void *w,
                                           int64_t N, int64_t Kw, int64_t ldw, uint8_t *qw,
                                           int64_t ldqw, float *sw, fp8bs_stream_t stream);

/* Normalization applied by fp8bs_norm_quantize_act_1x128. */
typedef enum { FP8BS_NORM_RMS = 0, FP8BS_NORM_LAYER = 1 } fp8bs_norm_kind;

/*
 * Normalization fused with the 1x128 activation cast -- "How I Improved My
 * Deepseek In In The Future", paragraph of hardware suggestions (fusion of
 * layer normalization and FP8 cast). Produces exactly what a normalization
 * layer with a bf16 output followed by fp8bs_quantize_act_1x128 produces,
 * without writing the normalized tensor to memory.
 *
 *   x      bf16  [M, K], row stride ldx (elements)            (input)
 *   gamma  bf16  [K]                                          (input)
 *   beta   bf16  [K] or NULL (no additive term)               (input)
 *   q      e4m3  [M, K], row stride ldq (bytes)               (output codes)
 *   scale  fp32  [M, K/128] row-major, contiguous             (output)
 *   mean   fp32  [M] or NULL; written for LayerNorm only      (output)
 *   rstd   fp32  [M] or NULL                                  (output)
 *
 * Per row, in binary32 with each step rounded to nearest:
 *   RMSNorm   (FP8BS_NORM_RMS):   mu = 0,       v = sum_k x^2 / K
 *   LayerNorm (FP8BS_NORM_LAYER): mu = sum_k x / K, v = sum_k (x - mu)^2 / K
 *   rstd = 1 / sqrt(v + eps)   (correctly rounded)
 *   y = bf16_rne(((x - mu) * rstd) * gamma + beta)
 * and then the 1x128 quantizer on y (codes and scales as in
 * fp8bs_quantize_act_1x128). The two sums are formed in a parallel order, so
 * mu and rstd may differ from a sequentially summed value by a few units in
 * the last place; given the returned mu and rstd, q and scale are exact.
 * K % 128 == 0 and 0 < K <= 65536 (else FP8BS_ERR_UNSUPPORTED; K == 0 with
 * M > 0 is FP8BS_ERR_INVALID_ARG); eps finite and >= 0 (eps == 0 with a
 * row whose v is 0 gives rstd = inf and non-finite y, outside the contract).
 * gamma and beta must be 16-byte aligned.
 */
fp8bs_status fp8bs_norm_quantize_act_1x128(const void *x, int64_t M, int64_t K, int64_t ldx,
                                           const void *gamma, const void *beta,
                                           fp8bs_norm_kind kind, float eps, uint8_t *q,
                                           int64_t ldq, float *scale, float *mean, float *rstd,
                                           fp8bs_stream_t stream);

/*
 * Weight quantization, 128x128 blocks (per 128 input x 128 output channels).
 *
 *   w      bf16  [N, K] (output channel x input channel), row stride ldw
 *   q      e4m3  [N, K], row stride ldq
 *   scale  fp32  [ceil(N/128), K/128] row-major, contiguous
 *
 * Block (nb, kb) covers rows 128nb..128nb+127 (only those < N) and columns
 * 128kb..128kb+127; its amax, scale and codes follow the same rule as the
 * activation tiles. K % 128 == 0 (else FP8BS_ERR_UNSUPPORTED). Stacked
 * expert weights [E, N, K] with N % 128 == 0 quantize as one [E*N, K] call.
 */
fp8bs_status fp8bs_quantize_weight_128x128(const void *w, int64_t N, int64_t K, int64_t ldw,
                                           uint8_t *q, int64_t ldq, float *scale,
                                           fp8bs_stream_t stream);

/*
 * Block-scaled FP8 GEMM: C[M, N] = A_hat * W_hat^T, where
 * A_hat[m, k] = decode(qa[m, k]) * sa[m, k/128] and
 * W_hat[n, k] = decode(qw[n, k]) * sw[n/128, k/128].
 *
 *   qa  e4m3 [M, K] contiguous          sa  fp32 [M, K/128] contiguous
 *   qw  e4m3 [N, K] contiguous          sw  fp32 [N/128, K/128] contiguous
 *   c   [M, N] with row stride ldc, fp32 or bf16 (RNE) per out_dtype
 *
 * Each 128-wide K chunk is multiplied on the tensor cores into an FP32
 * partial and then promoted: acc += sa[m, kb] * sw[n/128, kb] * partial.
 * Requires K % 128 == 0 and N % 128 == 0 (else FP8BS_ERR_UNSUPPORTED); any
 * M >= 0. K == 0 writes zeros. Accuracy: |C - C_exact| <=
 * 2e-5 * sum_k |A_hat W_hat| + 1e-6 (+ 2^-8 |C| for bf16 output).
 * The kernel runs one work unit (a CTA, or a CTA pair) per SM and deals the
 * output tiles out round by round. When the last round holds fewer tiles
 * than units (at most half as many), each of its tiles is cut into 2, 4 or
 * 8 column pieces of at least 32 columns computed by different units over
 * all K chunks; every output element keeps the same arithmetic, so the
 * result is that of an uncut launch bit for bit.
 */
fp8bs_status fp8bs_gemm(const uint8_t *qa, const float *sa, const uint8_t *qw, const float *sw,
                        void *c, fp8bs_out_dtype out_dtype, int64_t M, int64_t N, int64_t K,
                        int64_t ldc, fp8bs_stream_t stream);

/*
 * fp8bs_gemm with an explicit output tile (FP8BS_ERR_INVALID_ARG for an
 * unknown tile or PAIR_256x256 with N % 256 != 0).
 */
fp8bs_status fp8bs_gemm_tiled(const uint8_t *qa, const float *sa, const uint8_t *qw,
                              const float *sw, void *c, fp8bs_out_dtype out_dtype, int64_t M,
                              int64_t N, int64_t K, int64_t ldc, fp8bs_tile tile,
                              fp8bs_stream_t stream);

/*
 * fp8bs_gemm with a workspace that lets the GEMM balance its last wave of
 * output tiles. The kernel runs one work unit (a CTA, or a CTA pair for the
 * PAIR tiles) per SM and deals the tiles out round by round; when the tile
 * count is not a multiple of the unit count, the last round would leave most
 * units idle. With a workspace, each tile of that last round is instead cut
 * into S ranges of K chunks (S = min(units / tiles left, K / 2048), at least 2)
 * computed by different units: the owner of a tile (the unit with its first
 * range) adds the others' FP32 partial tiles, in range order, after its own
 * chunks, and stores C. Same output, same accuracy bound as fp8bs_gemm; the
 * bits of split tiles may differ from fp8bs_gemm's (the K sum is grouped
 * differently), but a given shape, tile and device always gives the same
 * bits.
 *
 *   workspace        DEVICE memory of at least the size
 *                    fp8bs_gemm_workspace_size reports, 256-byte aligned,
 *                    zero-filled before its first use (the kernel leaves it
 *                    reusable: flags it consumes are reset to zero). NULL:
 *                    no K split (exactly fp8bs_gemm_tiled, including its
 *                    column pieces). A shape whose last round cannot be
 *                    split along K is cut into column pieces instead.
 *   workspace_bytes  its size; too small: FP8BS_ERR_INVALID_ARG.
 * Two launches that use the same workspace at the same time on the GPU
 * (different streams) race; launches in one stream do not. The other
 * arguments are those of fp8bs_gemm_tiled. The library still allocates
 * nothing.
 */
fp8bs_status fp8bs_gemm_ws(const uint8_t *qa, const float *sa, const uint8_t *qw, const float *sw,
                           void *c, fp8bs_out_dtype out_dtype, int64_t M, int64_t N, int64_t K,
                           int64_t ldc, fp8bs_tile tile, void *workspace, size_t workspace_bytes,
                           fp8bs_stream_t stream);

/*
 * Workspace bytes fp8bs_gemm_ws needs for this shape and tile on the current
 * device (0 when no wave is split: the tile count is a multiple of the units,
 * K < 4096, or the problem fits in one partial wave). At most one FP32
 * 128 x 256 (or 128 x 128) tile per SM plus 32 bytes of flags per SM. Same
 * argument checks as fp8bs_gemm_tiled; bytes must not be NULL.
 */
fp8bs_status fp8bs_gemm_workspace_size(int64_t M, int64_t N, int64_t K, fp8bs_tile tile,
                                       size_t *bytes);

/*
 * fp8bs_gemm_ws for callers that cannot allocate device memory where they
 * call the GEMM: for example an allocator or memory-pool callback that must
 * not re-enter the allocator, a plug-in that may not own device memory, or
 * code on a path where cudaMalloc would synchronize the device or fail. The
 * pages describe no such call; it is an addition of this library.
 *
 * The workspace is a fixed 12 MiB (FP8BS_NOALLOC_SCRATCH_BYTES) array in the
 * library's own device memory: every GPU that loads the library holds it
 * until the process exits, and all calls on a device share it. The call
 * allocates and frees nothing (no cudaMalloc, no allocating library call).
 * Its first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it, so make that first call before any
 * stream capture. Calls whose executions overlap on the GPU (different
 * streams, or threads racing on one device) race on the shared array; calls
 * in one stream do not. A shape whose split needs more than the array
 * (fp8bs_gemm_workspace_size > FP8BS_NOALLOC_SCRATCH_BYTES) is rejected with
 * FP8BS_ERR_UNSUPPORTED before anything is launched; shapes that do not
 * split use no workspace. Arguments, results and accuracy are those of
 * fp8bs_gemm_ws; the bits equal fp8bs_gemm_ws's with any large enough
 * workspace.
 */
#define FP8BS_NOALLOC_SCRATCH_BYTES (12u << 20)
fp8bs_status fp8bs_gemm_noalloc(const uint8_t *qa, const float *sa, const uint8_t *qw,
                                const float *sw, void *c, fp8bs_out_dtype out_dtype, int64_t M,
                                int64_t N, int64_t K, int64_t ldc, fp8bs_tile tile,
                                fp8bs_stream_t stream);

/*
 * Grouped (MoE) GEMM: for each expert e, rows r in
 * [expert_offsets[e], expert_offsets[e+1]) of A are multiplied by W_e:
 * C[r, :] = A_hat[r, :] * W_hat_e^T.
 *
 *   qa, sa           as in fp8bs_gemm, with total_M rows
 *   expert_offsets   int32 [E+1], DEVICE memory: offsets[0] = 0,
 *                    nondecreasing, offsets[E] <= total_M. Read on the
 *                    device (no host synchronization); invalid offsets make
 *                    the kernel write nothing and are reported by
 *                    fp8bs_last_device_error as FP8BS_ERR_INVALID_ARG.
 *   qw               e4m3 [E, N, K] contiguous
 *   sw               fp32 [E, N/128, K/128] contiguous
 *   c                [total_M, N], row stride ldc; rows not covered by any
 *                    expert are left untouched
 *
 * 1 <= E <= 512; K % 128 == 0, N % 128 == 0. Same accuracy as fp8bs_gemm.
 */
fp8bs_status fp8bs_grouped_gemm(const uint8_t *qa, const float *sa, const int32_t *expert_offsets,
                                int32_t E, int64_t total_M, const uint8_t *qw, const float *sw,
                                void *c, fp8bs_out_dtype out_dtype, int64_t N, int64_t K,
                                int64_t ldc, fp8bs_stream_t stream);

/* fp8bs_grouped_gemm with an explicit output tile (see fp8bs_gemm_tiled). */
fp8bs_status fp8bs_grouped_gemm_tiled(const uint8_t *qa, const float *sa,
                                      const int32_t *expert_offsets, int32_t E, int64_t total_M,
                                      const uint8_t *qw, const float *sw, void *c,
                                      fp8bs_out_dtype out_dtype, int64_t N, int64_t K, int64_t ldc,
                                      fp8bs_tile tile, fp8bs_stream_t stream);

/*
 * The same GEMMs with the activation quantization fused in: A is given as
 * bf16 [M, K] (row stride lda elements, 16-byte aligned rows) and each
 * 1x128 tile is quantized inside the GEMM kernel -- loaded by TMA, scaled
 * and cast in shared memory, handed to the tensor cores -- so the E4M3 copy
 * of A and its scales never go to memory. This emulates in software the
 * fusion of the FP8 cast with the TMA load that "How I Improved My Deepseek
 * In In The Future" asks of future hardware (paragraph of hardware
 * suggestions). The codes and scales used are exactly those of
 * fp8bs_quantize_act_1x128, and the result is bit-identical to
 * fp8bs_quantize_act_1x128 followed by fp8bs_gemm_tiled /
 * fp8bs_grouped_gemm_tiled with FP8BS_TILE_128x256. W, its scales, C and the
 * remaining arguments are as in fp8bs_gemm / fp8bs_grouped_gemm.
 */
fp8bs_status fp8bs_gemm_bf16_act(const void *a, int64_t lda, const uint8_t *qw, const float *sw,
                                 void *c, fp8bs_out_dtype out_dtype, int64_t M, int64_t N,
                                 int64_t K, int64_t ldc, fp8bs_stream_t stream);

fp8bs_status fp8bs_grouped_gemm_bf16_act(const void *a, int64_t lda,
                                         const int32_t *expert_offsets, int32_t E,
                                         int64_t total_M, const uint8_t *qw, const float *sw,
                                         void *c, fp8bs_out_dtype out_dtype, int64_t N, int64_t K,
                                         int64_t ldc, fp8bs_stream_t stream);

/*
 * Fault injection for failure-detection tests; not for production use.
 * Every bounded wait of the GEMM kernels gives up after a limit (1 s by
 * default). With chunk >= 0, every later GEMM launch of this process (any of
 * the GEMM calls above, on any device) runs with waits limited to
 * wait_limit_ns, and the producer of its first CTA leaves out the copies of
 * its chunk number `chunk` (0-based over the 128-wide K chunks that CTA
 * loads), so the waits for that chunk run out: the kernel records
 * FP8BS_ERR_TIMEOUT for fp8bs_last_device_error, lets every copy it did
 * issue land, releases its tensor memory and returns; output tiles of that
 * CTA are left incomplete, nothing outside C is written. chunk < 0 restores
 * normal operation (default limit, nothing left out). 100 us <= wait_limit_ns
 * <= 10 s, chunk < 2^31, else FP8BS_ERR_INVALID_ARG. Not synchronized with
 * launches in flight on other threads.
 */
fp8bs_status fp8bs_test_inject_stall(int64_t chunk, int64_t wait_limit_ns);

/* Human-readable name of a status code (static string). */
const char *fp8bs_status_string(fp8bs_status status);

/*
 * Synchronizes `stream`, then reads and clears the current device's error
 * word: FP8BS_ERR_TIMEOUT if a bounded device wait expired since the last
 * call, FP8BS_ERR_INVALID_ARG if a grouped GEMM saw invalid offsets,
 * FP8BS_ERR_CUDA if the synchronization itself failed, else FP8BS_OK.
 * There is one error word per device, shared by every stream and thread:
 * kernels on other streams that have not finished are not waited for, and
 * an error they record later is reported by a later call. Only the bits that
 * were read are cleared (an atomic AND on `stream`), so no error recorded
 * between the read and the clear is lost.
 */
fp8bs_status fp8bs_last_device_error(fp8bs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
