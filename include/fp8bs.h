/*
 * fp8bs.h -- C ABI of libfp8bs: fine-grained FP8 (E4M3) quantization and block-scaled FP8
 * GEMM for NVIDIA B300 (sm_103a).
 *
 * The operations follow the DeepSeek-V3 FP8 training write-ups:
 *   [codingmall]  "Bạn có thể giải thích vai trò của độ chính xác FP8 trong quá trình đào tạo
 *                 của DeepSeek-V3" (codingmall.com), sections "Định lượng hạt mịn",
 *                 "Định lượng trực tuyến", "Tăng độ chính xác tích lũy", "Định dạng E4M3 hợp nhất";
 *   [dtcms]       DeepSeek-V3 overview (dtcms.com), section 三 "FP8混合精度训练", parts 1-3;
 *   [risenshine]  DeepSeek training-algorithm article (risenshineclean.com), section 三;
 *   [MoE]         dtcms.com section 一.2 "DeepSeekMoE架构" and risenshineclean.com section 二
 *                 (256 routed experts, each token routed to 8).
 * The pages define no interface; this one is the project's own.
 *
 * Conventions shared by every call
 *  - All tensors are row-major and live in DEVICE memory owned by the caller. The library
 *    never allocates per call; the first call on a device allocates one 4-byte error word that
 *    lives until the process exits (make that first call outside CUDA graph capture).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream) and
 *    never synchronize. Every output buffer is fully overwritten.
 *  - E4M3 codes are OCP E4M3FN bytes (bias 7, largest finite 448, no infinities).
 *  - Quantization of a tile with amax = max|x| > 0: s = amax / 448 (IEEE FP32 division),
 *    code = E4M3_rne_satfinite(x * (448 / amax)), one FP32 multiply per element; for
 *    amax < 2^-64 the same value is formed as (x * 2^64) * (448 / (amax * 2^64)). A tile with
 *    amax == 0 gets s = 1 and all codes 0x00. Dequantized value: decode(code) * s.
 *  - Argument errors are detected on the host before anything is launched and return
 *    FP8BS_ERR_INVALID_ARG or FP8BS_ERR_MISALIGNED; a device that is not sm_103 returns
 *    FP8BS_ERR_UNSUPPORTED_DEVICE; a CUDA launch error returns FP8BS_ERR_CUDA. Errors raised
 *    inside a running kernel (a pipeline wait that ran past its time budget) are reported
 *    later by fp8bs_last_error().
 *  - Calls are thread-safe. Non-finite inputs are outside the contract (no hang; the result
 *    is unspecified).
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *fp8bs_stream_t;

enum fp8bs_status {
    FP8BS_OK = 0,
    FP8BS_ERR_INVALID_ARG = -1,        /* shape, leading dimension, null pointer, dtype */
    FP8BS_ERR_MISALIGNED = -2,         /* a pointer or leading dimension breaks 16-byte alignment */
    FP8BS_ERR_UNSUPPORTED_DEVICE = -3, /* the current device is not compute capability 10.3 */
    FP8BS_ERR_CUDA = -4,               /* a CUDA runtime/driver call failed */
    FP8BS_ERR_TIMEOUT = -5             /* a kernel's pipeline wait ran past its budget */
};

enum fp8bs_out_dtype {
    FP8BS_OUT_BF16 = 0,
    FP8BS_OUT_F32 = 1
};

/*
 * Online 1x128 activation quantization ([codingmall] "Định lượng hạt mịn" and "Định lượng
 * trực tuyến"; [risenshine] 三: one token by 128 channels per tile).
 *   x       BF16 [M][ldx], the first K columns are read.
 *   q       E4M3 codes [M][ldq], the first K columns are written.
 *   scales  FP32 [K/128][M] (M contiguous): scales[kb*M + m] is the scale of row m, columns
 *           [128 kb, 128 kb + 128).
 * Requires M >= 0 (M == 0 is a no-op), K > 0, K % 128 == 0, ldx >= K, ldq >= K,
 * ldx % 8 == 0, ldq % 16 == 0, x and q 16-byte aligned, scales 4-byte aligned.
 */
int fp8_quant_act_1x128(const void *x, int64_t M, int64_t K, int64_t ldx,
                        uint8_t *q, int64_t ldq, float *scales, fp8bs_stream_t stream);

/*
 * Online 128x128 weight-block quantization ([codingmall] "Định lượng hạt mịn"; [dtcms] 三.2).
 *   w       BF16 [N][ldw] (row n is output channel n), the first K columns are read.
 *   q       E4M3 codes [N][ldq].
 *   scales  FP32 [ceil(N/128)][K/128]: scales[nb*(K/128) + kb] covers rows
 *           [128 nb, min(N, 128 nb + 128)) and columns [128 kb, 128 kb + 128). A last, partial
 *           row block takes its amax over its real rows only.
 * Stacked per-expert weights [E][N][K] with N % 128 == 0 may be passed as one [E*N][K]
 * matrix; the scales then come out as [E][N/128][K/128].
 * Requires N >= 0 (N == 0 is a no-op), K > 0, K % 128 == 0, ldw >= K, ldq >= K,
 * ldw % 8 == 0, ldq % 16 == 0, w and q 16-byte aligned, scales 4-byte aligned.
 */
int fp8_quant_weight_128x128(const void *w, int64_t N, int64_t K, int64_t ldw,
                             uint8_t *q, int64_t ldq, float *scales, fp8bs_stream_t stream);

/*
 * fp8_quant_act_1x128_ue8m0 / fp8_quant_weight_128x128_ue8m0: the same tiles, layouts and
 * requirements as fp8_quant_act_1x128 / fp8_quant_weight_128x128, with power-of-two scales.
 * This variant is not on the pages (their scale is amax/448); power-of-two (UE8M0) scales are
 * what Blackwell's block-scaled MMAs consume, and these calls let their numerics be compared:
 *   s = 2^e, e the smallest integer with 448 * 2^e >= amax (no value saturates), clamped below
 *   at e = -127; codes E4M3(x * 2^-e) (an exact scaling); a zero tile gets s = 1, codes 0x00.
 * The scales are ordinary FP32 values, so every GEMM call accepts them unchanged.
 */
int fp8_quant_act_1x128_ue8m0(const void *x, int64_t M, int64_t K, int64_t ldx,
                              uint8_t *q, int64_t ldq, float *scales, fp8bs_stream_t stream);
int fp8_quant_weight_128x128_ue8m0(const void *w, int64_t N, int64_t K, int64_t ldw,
                                   uint8_t *q, int64_t ldq, float *scales, fp8bs_stream_t stream);

/*
 * Block-scaled FP8 GEMM, C = A W^T ([dtcms] 三.1: FP8 inputs, BF16 or FP32 output;
 * [codingmall] "Tăng độ chính xác tích lũy": partial sums promoted to FP32 at intervals).
 *   C[m][n] = sum_kb  a_s[kb*M + m] * w_s[(n/128)*(K/128) + kb] * P[m][n][kb],
 *   P[m][n][kb] = sum over k in [128 kb, 128 kb + 128) of decode(a_q[m][k]) * decode(w_q[n][k]).
 * Each P is formed by the tensor cores in FP32 and promoted once per 128-wide K block: it is
 * multiplied by the FP32 product of its two scales and added to an FP32 accumulator with one
 * fused multiply-add. The accumulation order over K blocks is increasing kb. For M <= 64, when the
 * weight row tiles are too few to occupy the GPU, the K loop is cut into 2, 4 or 8 contiguous
 * ranges, each accumulated that way from zero, and their FP32 sums are added in range order; the
 * result depends only on M, N and K and the GPU's SM count (no atomics, deterministic).
 *   a_q  E4M3 [M][K] (contiguous rows), a_s FP32 [K/128][M]   (fp8_quant_act_1x128 layout)
 *   w_q  E4M3 [N][K] (contiguous rows), w_s FP32 [ceil(N/128)][K/128] (weight-quantizer layout)
 *   c    [M][ldc] of BF16 (out_dtype FP8BS_OUT_BF16, round to nearest even) or FP32.
 * Requires M >= 0 (M == 0 is a no-op), N > 0, N % 16 == 0, K > 0, K % 128 == 0,
 * M, N <= 2^31 - 1, ldc >= N, ldc * sizeof(out) % 16 == 0, a_q, w_q and c 16-byte aligned,
 * a_s and w_s 4-byte aligned.
 */
int fp8_blockscaled_gemm(const uint8_t *a_q, const float *a_s,
                         const uint8_t *w_q, const float *w_s,
                         int64_t M, int64_t N, int64_t K,
                         void *c, int64_t ldc, int out_dtype, fp8bs_stream_t stream);

/*
 * Grouped block-scaled FP8 GEMM for routed MoE experts ([MoE]; the pages name no grouped
 * kernel, this is the dense GEMM above applied per expert):
 *   for every group g and row r in [off[g], off[g+1]):
 *     C[r][n] = sum_kb a_s[kb*R + r] * w_s[g][n/128][kb] * P_g[r][n][kb]
 *   with P_g formed from a_q[r] and expert g's codes w_q[g][n].
 *   a_q            E4M3 [R][K], rows sorted by group; a_s FP32 [K/128][R]
 *   w_q            E4M3 [G][N][K]; w_s FP32 [G][ceil(N/128)][K/128]
 *   group_offsets  DEVICE int32 [G+1], off[0] = 0, non-decreasing, off[G] = R. The kernel
 *                  reads it on the device, so no host synchronization is needed. Offsets
 *                  outside [0, R] or decreasing are outside the contract (no hang; the rows
 *                  written are unspecified).
 *   c              [R][ldc] BF16 or FP32.
 * Requires G in [1, 1024], R >= 0 (R == 0 is a no-op), plus the dense call's rules for N, K,
 * ldc and alignment. Empty groups are allowed.
 */
int fp8_blockscaled_grouped_gemm(const uint8_t *a_q, const float *a_s,
                                 const uint8_t *w_q, const float *w_s,
                                 const int32_t *group_offsets, int64_t G, int64_t R,
                                 int64_t N, int64_t K, void *c, int64_t ldc, int out_dtype,
                                 fp8bs_stream_t stream);

/*
 * Grouped GEMM with a fused SwiGLU and 1x128 re-quantization of its output, for the expert FFN
 * (gate and up projections, then the down projection). The pages keep GEMM inputs in FP8,
 * accumulate in higher precision and convert back to FP8 for the next computation (szhzxw.cn
 * 一.2.c; [codingmall] "Định lượng trực tuyến": scales from the current tile maximum). The
 * activation between the two expert GEMMs is not on the pages; this call takes SwiGLU,
 * h = silu(gate) * up, DeepSeek-V3's expert FFN activation (a reading).
 *   w_q    E4M3 [G][N2][K] with gate and up rows interleaved in blocks of 128: rows
 *          [256 j, 256 j + 128) are the gate rows of channels [128 j, 128 j + 128) and rows
 *          [256 j + 128, 256 j + 256) their up rows; w_s FP32 [G][N2/128][K/128] as usual.
 *   a_q, a_s, group_offsets, G, R, K  as for fp8_blockscaled_grouped_gemm.
 *   h_q    E4M3 codes [R][ldh] of h, I = N2/2 channels per row (the A operand of the down GEMM)
 *   h_s    FP32 [I/128][R]: one scale per row and 128 channels (the 1x128 activation layout)
 * Per row r of group g: gate[c], up[c] = the block-scaled GEMM (FP32 accumulation as in
 * fp8_blockscaled_gemm) against expert g's gate/up rows of channel c; h[c] = fl(silu(gate[c]) *
 * up[c]) with silu(x) = x / (1 + e^-x) in FP32 from the fast exponential and division
 * intrinsics (__expf, __fdividef: a few ulps); then each 1x128 tile of h is quantized
 * exactly as fp8_quant_act_1x128 quantizes a tile (s = amax/448, codes E4M3(h * 448/amax)).
 * Requires N2 > 0, N2 % 256 == 0, ldh >= N2/2, ldh % 16 == 0, h_q 16-byte and h_s 4-byte
 * aligned, plus the grouped call's rules for the inputs. Rows outside every group are not
 * written.
 */
int fp8_blockscaled_grouped_gemm_swiglu_quant(const uint8_t *a_q, const float *a_s,
                                              const uint8_t *w_q, const float *w_s,
                                              const int32_t *group_offsets, int64_t G, int64_t R,
                                              int64_t N2, int64_t K, uint8_t *h_q, int64_t ldh,
                                              float *h_s, fp8bs_stream_t stream);

/*
 * MoE dispatch on the token side ([MoE]: each token is routed to 8 of 256 experts; the grouped
 * GEMMs read rows sorted by expert). The all-to-all between GPUs is not part of this library.
 *
 * fp8_moe_permute: gather token rows of quantized activations into the sorted row order.
 *   q             E4M3 codes [T][ldq] (K columns), s FP32 [K/128][T] (fp8_quant_act_1x128)
 *   token_of_row  DEVICE int32 [R]: sorted row r holds token token_of_row[r]
 *   qp            E4M3 codes [R][ldqp]: qp[r] = q[token_of_row[r]]
 *   sp            FP32 [K/128][R]: sp[kb][r] = s[kb][token_of_row[r]]
 * Bit copies. A token index outside [0, T) is outside the contract (that row is not written;
 * nothing faults). Requires T, R >= 0 (R == 0 is a no-op), K > 0, K % 128 == 0,
 * ldq, ldqp >= K and multiples of 16, q and qp 16-byte aligned, s, sp, token_of_row 4-byte.
 */
int fp8_moe_permute(const uint8_t *q, int64_t ldq, const float *s, int64_t T,
                    const int32_t *token_of_row, int64_t R, int64_t K, uint8_t *qp, int64_t ldqp,
                    float *sp, fp8bs_stream_t stream);

/*
 * fp8_moe_combine: each token's output is the routing-weighted sum of its expert rows,
 *   out[t][n] = sum_j weights[t][j] * y[row_of_token[t][j]][n],
 * accumulated in FP32 as acc = fma(weights[t][j], y, acc) for j = 0 .. topk-1 in order from 0,
 * then rounded to BF16 (nearest, ties to even).
 *   y             BF16 [R][ldy] (N columns): the expert outputs in sorted row order
 *   row_of_token  DEVICE int32 [T][topk]; weights DEVICE FP32 [T][topk]
 *   out           BF16 [T][ldo]
 * A row index outside [0, R) adds nothing (outside the contract). Requires T >= 0 (T == 0 is a
 * no-op), 1 <= topk <= 32, N > 0, N % 8 == 0, ldy, ldo >= N and multiples of 8, y and out
 * 16-byte aligned, row_of_token and weights 4-byte aligned.
 */
int fp8_moe_combine(const void *y, int64_t ldy, int64_t R, const int32_t *row_of_token,
                    const float *weights, int64_t T, int64_t topk, int64_t N, void *out,
                    int64_t ldo, fp8bs_stream_t stream);

/*
 * Backward pass. The pages use the same E4M3 format in the backward pass as in the forward
 * pass ([codingmall] "Định dạng E4M3 hợp nhất"; [dtcms] 三.2) and name no backward tile shapes.
 * Reading: a block-scaled contraction needs one scale per 128-long block of the contracted
 * index, so
 *   data gradient    dX[M][K] = dY[M][N] W[N][K]: fp8_quant_act_1x128 on dY, W as W^T codes
 *                    in its 128x128 blocks (fp8_quant_weight_128x128_t), fp8_blockscaled_gemm;
 *   weight gradient  dW[N][K] = dY^T X (contracting over the M tokens): dY and X in 128x1 tiles
 *                    (fp8_quant_act_128x1), fp8_blockscaled_gemm_1d1d.
 */

/*
 * 128x1 tiles: one scale per 128 consecutive rows of one column (128 tokens of one channel),
 * with the codes written transposed so that the rows become the contiguous, contracted index.
 *   x       BF16 [M][ldx], the first K columns are read.
 *   qt      E4M3 codes [K][ldqt]: qt[k*ldqt + m] is the code of x[m][k].
 *   scales  FP32 [M/128][K]: scales[mb*K + k] covers rows [128 mb, 128 mb + 128) of column k
 *           (the a_s / b_s layout fp8_blockscaled_gemm_1d1d expects for an operand qt).
 * Tile arithmetic as for every quantizer above. Requires M >= 0 (M == 0 is a no-op),
 * M % 128 == 0, M / 128 <= 65535, K > 0, K % 128 == 0, ldx >= K, ldqt >= M, ldx % 8 == 0,
 * ldqt % 16 == 0, x and qt 16-byte aligned, scales 4-byte aligned.
 */
int fp8_quant_act_128x1(const void *x, int64_t M, int64_t K, int64_t ldx,
                        uint8_t *qt, int64_t ldqt, float *scales, fp8bs_stream_t stream);

/*
 * 128x128 weight blocks with the codes written as W^T, the B operand of the data-gradient GEMM
 * (which contracts over N). The blocks, their scales and their codes are exactly those of
 * fp8_quant_weight_128x128 on the same W; only the layout differs.
 *   w         BF16 [N][ldw], the first K columns are read.
 *   qt        E4M3 codes [K][ldqt]: qt[k*ldqt + n] is the code of w[n][k].
 *   scales_t  FP32 [K/128][N/128]: scales_t[kb*(N/128) + nb] is the scale of block (nb, kb)
 *             (the w_s layout fp8_blockscaled_gemm expects for a weight operand qt [K][N]).
 * Requires N >= 0 (N == 0 is a no-op), N % 128 == 0, N / 128 <= 65535, K > 0, K % 128 == 0,
 * ldw >= K, ldqt >= N, ldw % 8 == 0, ldqt % 16 == 0, w and qt 16-byte aligned, scales_t
 * 4-byte aligned.
 */
int fp8_quant_weight_128x128_t(const void *w, int64_t N, int64_t K, int64_t ldw,
                               uint8_t *qt, int64_t ldqt, float *scales_t, fp8bs_stream_t stream);

/*
 * Block-scaled FP8 GEMM with a per-row scale on both operands ("1d1d"; the weight-gradient
 * GEMM), C = A B^T:
 *   C[m][n] = sum_kb a_s[kb*M + m] * b_s[kb*N + n] * P[m][n][kb],
 *   P[m][n][kb] = sum over k in [128 kb, 128 kb + 128) of decode(a_q[m][k]) * decode(b_q[n][k]).
 * P is formed by the tensor cores in FP32 and promoted once per K block in FP32:
 * acc = fma(P * b_s[kb][n], a_s[kb][m], acc), increasing kb.
 *   a_q  E4M3 [M][K] (contiguous rows), a_s FP32 [K/128][M]
 *   b_q  E4M3 [N][K] (contiguous rows), b_s FP32 [K/128][N]
 *   c    [M][ldc] BF16 or FP32, as for fp8_blockscaled_gemm.
 * For dW = dY^T X: a = fp8_quant_act_128x1(dY) (M = channels of dY), b = fp8_quant_act_128x1(X)
 * (N = channels of X), K = tokens. Requirements as for fp8_blockscaled_gemm.
 */
int fp8_blockscaled_gemm_1d1d(const uint8_t *a_q, const float *a_s,
                              const uint8_t *b_q, const float *b_s,
                              int64_t M, int64_t N, int64_t K,
                              void *c, int64_t ldc, int out_dtype, fp8bs_stream_t stream);

/*
 * fp8_blockscaled_gemm_quant: fp8_blockscaled_gemm with its output re-quantized to E4M3 in 1x128
 * tiles in the epilogue, ready to be the next GEMM's A operand. The pages accumulate in higher
 * precision and convert back to FP8 for the next computation (szhzxw.cn 一.2.c), with the
 * scales from each tile's current maximum ([codingmall] "Định lượng trực tuyến").
 * Per row m and 128 output columns [128 j, 128 j + 128): the FP32 results C[m][n] (accumulated
 * exactly as fp8_blockscaled_gemm accumulates them) form one tile, quantized as
 * fp8_quant_act_1x128 quantizes a tile (s = amax/448, codes E4M3(C * 448/amax), the same tiny
 * and zero rules).
 *   c_q  E4M3 codes [M][ldcq]; c_s FP32 [N/128][M] (c_s[j*M + m]).
 * Inputs and their requirements as for fp8_blockscaled_gemm, plus N % 128 == 0, ldcq >= N,
 * ldcq % 16 == 0, c_q 16-byte and c_s 4-byte aligned. Runs on the tiled CTA-pair kernel for
 * every M.
 */
int fp8_blockscaled_gemm_quant(const uint8_t *a_q, const float *a_s,
                               const uint8_t *w_q, const float *w_s,
                               int64_t M, int64_t N, int64_t K,
                               uint8_t *c_q, int64_t ldcq, float *c_s, fp8bs_stream_t stream);

/*
 * fp8_blockscaled_gemm_noalloc: the same dense block-scaled GEMM as fp8_blockscaled_gemm, for
 * callers that cannot let a library allocate device memory. The pages describe no such interface;
 * this entry point has no counterpart there.
 *
 * Who needs it: frameworks that hand out all device memory through their own caching allocator
 * or pool and treat any cudaMalloc behind its back as an error (it would fragment or exceed the
 * pool's budget), and deployments that must fix their device footprint before they start.
 * fp8_blockscaled_gemm allocates a 4-byte error word with cudaMalloc on its first call on a
 * device; this variant never calls cudaMalloc, cudaFree or any allocating routine.
 *
 * Instead its kernels keep that scratch word in a fixed 256-byte array inside the library image
 * (a static __device__ array: every GPU that loads the library holds it until the process exits).
 * A call needs one 4-byte word of it for any problem size; a call that would need more than the
 * array holds is rejected with FP8BS_ERR_INVALID_ARG before anything is launched.
 *
 * The first call on a device looks up the array's device address (once per device, with that
 * device current); make that first call before any stream capture begins. Every call shares the
 * same array and it keeps what the last call left there: the word is zero when the library is
 * loaded, a kernel only ever moves it from zero to a timeout code, and fp8bs_last_error() reads
 * it (beside the regular error word) and sets it back to zero, so a timeout stays recorded until
 * it is read. Calls that can overlap on the GPU (different streams without ordering between them)
 * race on that word, and a recorded timeout cannot then be attributed to one of them: order them.
 *
 * Dispatch, arguments, layouts, requirements and results are exactly those of
 * fp8_blockscaled_gemm (the few-row kernel for M <= 64, the CTA-pair kernel above), so the two
 * calls return identical outputs.
 */
int fp8_blockscaled_gemm_noalloc(const uint8_t *a_q, const float *a_s,
                                 const uint8_t *w_q, const float *w_s,
                                 int64_t M, int64_t N, int64_t K,
                                 void *c, int64_t ldc, int out_dtype, fp8bs_stream_t stream);

/*
 * Test hook for failure detection (not for production use): the next grouped GEMM launch
 * (fp8_blockscaled_grouped_gemm) runs with one epilogue warp skipping its release of the TMEM
 * accumulator at accumulation step `at` (0-based over the CTA's K blocks). A release that never
 * comes makes the MMA issuer's wait run past its budget; the kernel then records
 * FP8BS_ERR_TIMEOUT, every role stops and drains its in-flight copies and MMAs, and the kernel
 * returns, so the CUDA context stays usable. One-shot: later launches are unaffected.
 * Returns FP8BS_ERR_INVALID_ARG for at < 0.
 */
int fp8bs_debug_skip_release(int at);

/* Human-readable name of a status code. The string is static. */
const char *fp8bs_status_string(int status);

/*
 * Synchronizes `stream`, then reads and clears the current device's error words: the one the
 * GEMM kernels set when a pipeline wait runs past its budget (they then stop, drain their
 * in-flight copies and return), and the one inside the library image that
 * fp8_blockscaled_gemm_noalloc's kernels use. Allocates nothing. Returns FP8BS_OK,
 * FP8BS_ERR_TIMEOUT (either word recorded a timeout) or FP8BS_ERR_CUDA.
 */
int fp8bs_last_error(fp8bs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
