/* A plain C99 client of include/fp8bs.h: the header must compile as C, every declared call must
 * link against libfp8bs.so, and argument errors must come back from the host-side checks
 * (fake, never-dereferenced pointers; no device is touched). Prints one line per check and
 * exits with the number of failures. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "fp8bs.h"

static int failures = 0;

static void expect(const char *what, int got, int want)
{
    const int ok = got == want;
    printf("%s %s: got %d (%s), want %d\n", ok ? "ok  " : "FAIL", what, got,
           fp8bs_status_string(got), want);
    failures += !ok;
}

int main(void)
{
    uint8_t *const q = (uint8_t *)(uintptr_t)0x1000;
    const void *const x = (const void *)(uintptr_t)0x2000;
    float *const s = (float *)(uintptr_t)0x3004;
    const int32_t *const off = (const int32_t *)(uintptr_t)0x4000;

    expect("status string of OK", strcmp(fp8bs_status_string(FP8BS_OK), "FP8BS_OK"), 0);
    expect("act 1x128, K not a multiple of 128",
           fp8_quant_act_1x128(x, 4, 100, 128, q, 128, s, NULL), FP8BS_ERR_INVALID_ARG);
    expect("act 1x128, misaligned input",
           fp8_quant_act_1x128((const char *)x + 2, 4, 128, 128, q, 128, s, NULL),
           FP8BS_ERR_MISALIGNED);
    expect("weight 128x128, null codes",
           fp8_quant_weight_128x128(x, 128, 128, 128, NULL, 128, s, NULL), FP8BS_ERR_INVALID_ARG);
    expect("act 128x1, rows not a multiple of 128",
           fp8_quant_act_128x1(x, 100, 128, 128, q, 128, s, NULL), FP8BS_ERR_INVALID_ARG);
    expect("weight 128x128 transposed, ld < K",
           fp8_quant_weight_128x128_t(x, 128, 256, 128, q, 128, s, NULL), FP8BS_ERR_INVALID_ARG);
    expect("gemm, bad output dtype",
           fp8_blockscaled_gemm(q, s, q, s, 16, 128, 128, q, 128, 7, NULL),
           FP8BS_ERR_INVALID_ARG);
    expect("gemm, N not a multiple of 16",
           fp8_blockscaled_gemm(q, s, q, s, 16, 100, 128, q, 128, FP8BS_OUT_BF16, NULL),
           FP8BS_ERR_INVALID_ARG);
    expect("gemm 1d1d, K not a multiple of 128",
           fp8_blockscaled_gemm_1d1d(q, s, q, s, 16, 128, 100, q, 128, FP8BS_OUT_F32, NULL),
           FP8BS_ERR_INVALID_ARG);
    expect("grouped gemm, no groups",
           fp8_blockscaled_grouped_gemm(q, s, q, s, off, 0, 128, 128, 128, q, 128,
                                        FP8BS_OUT_BF16, NULL),
           FP8BS_ERR_INVALID_ARG);
    expect("gemm with re-quantized output, N not a multiple of 128",
           fp8_blockscaled_gemm_quant(q, s, q, s, 256, 144, 128, q, 144, s, NULL),
           FP8BS_ERR_INVALID_ARG);
    expect("moe permute, negative rows",
           fp8_moe_permute(q, 128, s, 4, off, -1, 128, q, 128, s, NULL), FP8BS_ERR_INVALID_ARG);
    printf("%d failure(s)\n", failures);
    return failures;
}
