/*
 * fp8_oracle.c -- plain, slow CPU oracle for fine-grained FP8 quantization and the
 * block-scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the package smoke check and the benchmark's CPU
 * baseline load this file (as liboracle.so, through oracle/oracle.py). The CUDA library
 * shares no code, header, table or constant with it, and the product path never calls it.
 *
 * What it follows (the pages describe the method in words only; no listing is used):
 *  [codingmall] "Bạn có thể giải thích vai trò của độ chính xác FP8 trong quá trình đào tạo
 *      của DeepSeek-V3", sections "Định lượng hạt mịn" (activations grouped in 1x128 tiles,
 *      weights in 128x128 blocks, each scaled on its own), "Định lượng trực tuyến" (the
 *      scale of a tile comes from that tile's current maximum, not from a history),
 *      "Tăng độ chính xác tích lũy" (partial sums promoted to FP32 at intervals during the
 *      GEMM) and "Định dạng E4M3 hợp nhất" (E4M3 for every FP8 tensor).
 *  [dtcms] DeepSeek-V3 overview, section 三 "FP8混合精度训练", parts 1-3: GEMMs take FP8
 *      inputs and produce BF16 or FP32; 1x128 tile / 128x128 block grouping; accumulation
 *      raised in precision.
 *  [risenshine] DeepSeek training-algorithm article, section 三: a 1x128 tile is one token
 *      by 128 channels; partial results are periodically promoted to FP32 registers.
 *
 * Readings where the pages are silent (each one is also listed in the design notes):
 *  - E4M3 is the OCP "E4M3FN" layout: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
 *    no infinities, S.1111.111 is NaN, largest finite value 448.
 *  - Encoding rounds to nearest, ties to even mantissa, and saturates to +-448.
 *    A result that rounds to zero keeps the sign of its input.
 *  - Scale of a tile with amax > 0: s = amax / 448 (one IEEE FP32 division); the values are
 *    encoded as E4M3(x * r) with r = 448 / amax (a second IEEE FP32 division), one FP32
 *    multiply per element. For amax < 2^-64, r would overflow for the smallest amax, so the
 *    same quantity is formed as r = 448 / (amax * 2^64) and E4M3((x * 2^64) * r); both
 *    power-of-two scalings are exact, so the result is the one the plain formula gives with
 *    an unbounded exponent range.
 *  - A tile whose amax is 0 gets s = 1 and all codes 0x00.
 *  - The promotion interval is one 128-wide K block: the scales change every 128 K, so a
 *    partial cannot be promoted less often.
 *  - Scale layouts: activation scales [K/128][M] (M contiguous); weight scales
 *    [ceil(N/128)][K/128] (K blocks contiguous). A last, partial weight block's amax covers
 *    only its real rows.
 *  - Backward pass ([codingmall] "Định dạng E4M3 hợp nhất", [dtcms] 三.2: the same E4M3
 *    format for the backward pass). The pages name no backward tile shapes. A block-scaled
 *    contraction needs one scale per 128-long block of the contracted index, so:
 *      dgrad dX = dY W    contracts over N: dY in 1x128 tiles (the forward quantizer), W in
 *                         its 128x128 blocks, its codes laid out as W^T [K][N];
 *      wgrad dW = dY^T X  contracts over the M tokens: dY and X in 128x1 tiles (128 tokens of
 *                         one channel), codes laid out transposed [channels][M], and the GEMM
 *                         takes a per-row scale on both operands ("1d1d").
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------------------ */
/* BF16 and E4M3 from their bit definitions                                               */
/* ------------------------------------------------------------------------------------ */

/* A BF16 value is the top 16 bits of an IEEE binary32; widening is exact. */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a finite binary32 to BF16, nearest with ties to even: add 0x7FFF plus the kept part's
 * lowest bit to the bit pattern and truncate (a carry into the exponent is the correct
 * rounding up). Non-finite values are outside the contract. */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t b;
    memcpy(&b, &f, 4);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

/* Value of one E4M3FN code: sign s, biased exponent e (bias 7), mantissa m.
 * e == 0 is subnormal: m * 2^-9. Otherwise (1 + m/8) * 2^(e-7). S.1111.111 is NaN. */
double orc_e4m3_decode(uint8_t code)
{
    int s = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round p to the nearest E4M3FN value, ties to even mantissa, saturating at +-448.
 * NaN input is outside the contract. */
uint8_t orc_e4m3_encode(float p)
{
    uint8_t sign = signbit(p) ? 0x80 : 0x00;
    double a = fabs((double)p);
    double t;
    int e2, E, eb;

    if (a >= 448.0)                       /* saturate (covers the 464 midpoint and inf) */
        return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {             /* subnormal range: grid step 2^-9 */
        t = rint(ldexp(a, 9));            /* exact scaling, then ties-to-even */
        return sign | (uint8_t)t;         /* t == 8 is code 0x08, the smallest normal */
    }
    (void)frexp(a, &e2);                  /* a = f * 2^e2 with f in [0.5, 1) */
    E = e2 - 1;                           /* a = (1 + mant) * 2^E */
    t = rint((ldexp(a, -E) - 1.0) * 8.0); /* mantissa in steps of 1/8, ties-to-even */
    if (t == 8.0) {                       /* rounded up to the next power of two */
        t = 0.0;
        E += 1;
    }
    eb = E + 7;
    if (eb > 15 || (eb == 15 && t == 7.0)) /* unreachable for a < 448; kept as a guard */
        return sign | 0x7E;
    return sign | (uint8_t)((eb << 3) | (int)t);
}

void orc_e4m3_encode_array(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_e4m3_encode(x[i]);
}

void orc_e4m3_decode_array(const uint8_t *c, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------------------------ */
/* Online tile scaling ([codingmall] "Định lượng trực tuyến")                             */
/* ------------------------------------------------------------------------------------ */

typedef struct {
    float s;     /* dequantization scale: x ~ decode(q) * s */
    float r;     /* quantization multiplier */
    int tiny;    /* 1: amax < 2^-64, use the exact power-of-two rewrite */
    int zero;    /* 1: amax == 0 */
} tile_scale_t;

static tile_scale_t tile_scale(float amax)
{
    tile_scale_t t;
    t.tiny = 0;
    t.zero = 0;
    if (amax == 0.0f) {
        t.s = 1.0f;
        t.r = 0.0f;
        t.zero = 1;
        return t;
    }
    t.s = amax / 448.0f;
    if (amax < 0x1p-64f) {
        t.r = 448.0f / (amax * 0x1p64f);
        t.tiny = 1;
    } else {
        t.r = 448.0f / amax;
    }
    return t;
}

/* Power-of-two (UE8M0) tile scale, a variant that is not on the pages (Blackwell's block-scaled
 * MMAs take such scales): s = 2^e with e the smallest integer for which 448 * 2^e >= amax, so that
 * no value saturates, clamped below at UE8M0's 2^-127; codes E4M3(x * 2^-e), an exact scaling.
 * With amax = f * 2^E (frexp, f in [0.5, 1)) and 448 = 0.875 * 2^9, e = E - 9 + (f > 0.875). */
static int ue8m0_exponent(float amax)
{
    int E;
    float f = frexpf(amax, &E);
    int e = E - 9 + (f > 0.875f ? 1 : 0);
    return e < -127 ? -127 : e;
}

static tile_scale_t tile_scale_ue8m0(float amax)
{
    tile_scale_t t;
    t.tiny = 0;
    t.zero = 0;
    if (amax == 0.0f) {
        t.s = 1.0f;
        t.r = 0.0f;
        t.zero = 1;
        return t;
    }
    int e = ue8m0_exponent(amax);
    t.s = ldexpf(1.0f, e);
    t.r = ldexpf(1.0f, -e);
    return t;
}

int orc_ue8m0_exponent(float amax) { return ue8m0_exponent(amax); }

static uint8_t tile_encode(float x, const tile_scale_t *t)
{
    float y;
    if (t->zero)
        return 0x00;
    y = t->tiny ? (x * 0x1p64f) * t->r : x * t->r;
    return orc_e4m3_encode(y);
}

/* 1x128 activation tiles: one scale per row m and 128-column block kb.
 * x: BF16 bits [M][ldx]; q: codes [M][ldq]; s: [K/128][M]. K must be a multiple of 128. */
static void quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                            uint8_t *q, int64_t ldq, float *s, int ue8m0)
{
    int64_t KB = K / 128;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t kb = 0; kb < KB; kb++) {
            const uint16_t *xt = x + m * ldx + kb * 128;
            uint8_t *qt = q + m * ldq + kb * 128;
            float amax = 0.0f;
            tile_scale_t t;
            for (int k = 0; k < 128; k++)
                amax = fmaxf(amax, fabsf(bf16_bits_to_float(xt[k])));
            t = ue8m0 ? tile_scale_ue8m0(amax) : tile_scale(amax);
            for (int k = 0; k < 128; k++)
                qt[k] = tile_encode(bf16_bits_to_float(xt[k]), &t);
            s[kb * M + m] = t.s;
        }
    }
}

void orc_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                         uint8_t *q, int64_t ldq, float *s)
{
    quant_act_1x128(x, M, K, ldx, q, ldq, s, 0);
}

/* The same tiles with power-of-two scales (tile_scale_ue8m0). */
void orc_quant_act_1x128_ue8m0(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                               uint8_t *q, int64_t ldq, float *s)
{
    quant_act_1x128(x, M, K, ldx, q, ldq, s, 1);
}

/* 128x128 weight blocks: one scale per (128 rows of N) x (128 columns of K).
 * w: BF16 bits [N][ldw]; q: codes [N][ldq]; s: [ceil(N/128)][K/128].
 * The last row block may be partial; its amax covers only rows < N. */
static void quant_weight_128x128(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                                 uint8_t *q, int64_t ldq, float *s, int ue8m0)
{
    int64_t KB = K / 128;
    int64_t NB = (N + 127) / 128;
    for (int64_t nb = 0; nb < NB; nb++) {
        int64_t n_end = (nb + 1) * 128 < N ? (nb + 1) * 128 : N;
        for (int64_t kb = 0; kb < KB; kb++) {
            float amax = 0.0f;
            tile_scale_t t;
            for (int64_t n = nb * 128; n < n_end; n++)
                for (int k = 0; k < 128; k++)
                    amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[n * ldw + kb * 128 + k])));
            t = ue8m0 ? tile_scale_ue8m0(amax) : tile_scale(amax);
            for (int64_t n = nb * 128; n < n_end; n++)
                for (int k = 0; k < 128; k++)
                    q[n * ldq + kb * 128 + k] =
                        tile_encode(bf16_bits_to_float(w[n * ldw + kb * 128 + k]), &t);
            s[nb * KB + kb] = t.s;
        }
    }
}

void orc_quant_weight_128x128(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                              uint8_t *q, int64_t ldq, float *s)
{
    quant_weight_128x128(w, N, K, ldw, q, ldq, s, 0);
}

/* The same blocks with power-of-two scales (tile_scale_ue8m0). */
void orc_quant_weight_128x128_ue8m0(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                                    uint8_t *q, int64_t ldq, float *s)
{
    quant_weight_128x128(w, N, K, ldw, q, ldq, s, 1);
}

/* 128x1 activation tiles for the weight-gradient GEMM: one scale per 128 consecutive rows
 * (tokens) of one column (channel). x: BF16 bits [M][ldx]; the codes are written transposed,
 * qt[k][m] at qt + k*ldqt + m (so the tokens become the contiguous, contracted index); scales
 * s[mb][k] at s + mb*K + k. M must be a multiple of 128. */
void orc_quant_act_128x1(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                         uint8_t *qt, int64_t ldqt, float *s)
{
    int64_t MB = M / 128;
    for (int64_t k = 0; k < K; k++) {
        for (int64_t mb = 0; mb < MB; mb++) {
            float amax = 0.0f;
            tile_scale_t t;
            for (int i = 0; i < 128; i++)
                amax = fmaxf(amax, fabsf(bf16_bits_to_float(x[(mb * 128 + i) * ldx + k])));
            t = tile_scale(amax);
            for (int i = 0; i < 128; i++)
                qt[k * ldqt + mb * 128 + i] =
                    tile_encode(bf16_bits_to_float(x[(mb * 128 + i) * ldx + k]), &t);
            s[mb * K + k] = t.s;
        }
    }
}

/* 128x128 weight blocks with the codes written transposed, for the data-gradient GEMM that
 * contracts over N: qt[k][n] at qt + k*ldqt + n, scales st[kb][nb] at st + kb*(N/128) + nb.
 * The blocks, their amax and their codes are those of the forward weight quantizer.
 * N and K must be multiples of 128. */
void orc_quant_weight_128x128_t(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                                uint8_t *qt, int64_t ldqt, float *st)
{
    int64_t KB = K / 128;
    int64_t NB = N / 128;
    for (int64_t nb = 0; nb < NB; nb++) {
        for (int64_t kb = 0; kb < KB; kb++) {
            float amax = 0.0f;
            tile_scale_t t;
            for (int64_t n = nb * 128; n < nb * 128 + 128; n++)
                for (int64_t k = kb * 128; k < kb * 128 + 128; k++)
                    amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[n * ldw + k])));
            t = tile_scale(amax);
            for (int64_t n = nb * 128; n < nb * 128 + 128; n++)
                for (int64_t k = kb * 128; k < kb * 128 + 128; k++)
                    qt[k * ldqt + n] = tile_encode(bf16_bits_to_float(w[n * ldw + k]), &t);
            st[kb * NB + nb] = t.s;
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* Block-scaled GEMM: C = A * W^T on the quantized operands                               */
/*   C[m,n] = sum_kb s_a[kb][m] * s_w[n/128][kb] * sum_{k in kb} dec(a[m,k]) * dec(w[n,k])  */
/* ([dtcms] 三.1 and 三.3, [codingmall] "Tăng độ chính xác tích lũy")                     */
/* ------------------------------------------------------------------------------------ */

/* Value of every code, filled per call (callers may run on several threads). */
static void dec_table(double dec[256])
{
    for (int c = 0; c < 256; c++)
        dec[c] = orc_e4m3_decode((uint8_t)c);
}

/* One output element in FP64. Every E4M3 product and every 128-term block sum is exact in
 * FP64, so the only roundings are the scale products and the sum over K blocks.
 * *abs_out gets sum_k |a_hat_k * w_hat_k| (dequantized operands), the error-bound weight. */
static double point_f64(const double *dec,
                        const uint8_t *arow, const float *as, int64_t as_ld, int64_t m,
                        const uint8_t *wrow, const float *ws_row, int64_t ws_step, int64_t KB,
                        double *abs_out)
{
    double c = 0.0, cabs = 0.0;
    for (int64_t kb = 0; kb < KB; kb++) {
        double part = 0.0, part_abs = 0.0;
        double sc = (double)as[kb * as_ld + m] * (double)ws_row[kb * ws_step];
        for (int k = 0; k < 128; k++) {
            double p = dec[arow[kb * 128 + k]] * dec[wrow[kb * 128 + k]];
            part += p;
            part_abs += fabs(p);
        }
        c += sc * part;
        cabs += fabs(sc) * part_abs;
    }
    if (abs_out)
        *abs_out = cabs;
    return c;
}

/* The same element with an FP32 partial per K block (sequential, products exact in FP32)
 * and an FP32 fused multiply-add promotion: acc = fma(partial, s_a * s_w, acc).
 * ws_row[kb * ws_step] is the second operand's scale of K block kb (step 1 for a weight
 * block row, N for per-row scales [K/128][N]). */
static float point_f32(const double *dec, const uint8_t *arow, const float *as, int64_t as_ld, int64_t m,
                       const uint8_t *wrow, const float *ws_row, int64_t ws_step, int64_t KB)
{
    float acc = 0.0f;
    for (int64_t kb = 0; kb < KB; kb++) {
        float part = 0.0f;
        float sc = as[kb * as_ld + m] * ws_row[kb * ws_step];
        for (int k = 0; k < 128; k++)
            part += (float)dec[arow[kb * 128 + k]] * (float)dec[wrow[kb * 128 + k]];
        acc = fmaf(part, sc, acc);
    }
    return acc;
}

/* Selected elements (pm[i], pn[i]) of the dense GEMM.
 * aq [M][lda] codes, as [K/128][M]; wq [N][ldw] codes, ws [ceil(N/128)][K/128].
 * out_f64 / out_abs / out_f32 may each be NULL. */
void orc_gemm_points(const uint8_t *aq, int64_t lda, const float *as,
                     const uint8_t *wq, int64_t ldw, const float *ws,
                     int64_t M, int64_t N, int64_t K,
                     int64_t npts, const int64_t *pm, const int64_t *pn,
                     double *out_f64, double *out_abs, float *out_f32)
{
    int64_t KB = K / 128;
    (void)N;
    double dec[256];
    dec_table(dec);
    for (int64_t i = 0; i < npts; i++) {
        int64_t m = pm[i], n = pn[i];
        const uint8_t *arow = aq + m * lda;
        const uint8_t *wrow = wq + n * ldw;
        const float *ws_row = ws + (n / 128) * KB;
        double cabs;
        double c = point_f64(dec, arow, as, M, m, wrow, ws_row, 1, KB, &cabs);
        if (out_f64)
            out_f64[i] = c;
        if (out_abs)
            out_abs[i] = cabs;
        if (out_f32)
            out_f32[i] = point_f32(dec, arow, as, M, m, wrow, ws_row, 1, KB);
    }
}

/* Whole output, C64 [M][N] and its bound weight Cabs [M][N] (either may be NULL). */
void orc_gemm_f64(const uint8_t *aq, int64_t lda, const float *as,
                  const uint8_t *wq, int64_t ldw, const float *ws,
                  int64_t M, int64_t N, int64_t K, double *c, double *cabs)
{
    int64_t KB = K / 128;
    double dec[256];
    dec_table(dec);
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            double ab;
            double v = point_f64(dec, aq + m * lda, as, M, m, wq + n * ldw, ws + (n / 128) * KB,
                                 1, KB, &ab);
            if (c)
                c[m * N + n] = v;
            if (cabs)
                cabs[m * N + n] = ab;
        }
}

/* GEMM with a per-row scale on both operands ("1d1d", the weight-gradient GEMM):
 *   C[m,n] = sum_kb s_a[kb][m] * s_b[kb][n] * sum_{k in kb} dec(a[m,k]) * dec(b[n,k]).
 * aq [M][lda], as [K/128][M]; bq [N][ldb], bs [K/128][N]. Selected elements (pm[i], pn[i]);
 * out_f64 / out_abs / out_f32 may each be NULL. */
void orc_gemm_1d1d_points(const uint8_t *aq, int64_t lda, const float *as,
                          const uint8_t *bq, int64_t ldb, const float *bs,
                          int64_t M, int64_t N, int64_t K,
                          int64_t npts, const int64_t *pm, const int64_t *pn,
                          double *out_f64, double *out_abs, float *out_f32)
{
    int64_t KB = K / 128;
    double dec[256];
    dec_table(dec);
    for (int64_t i = 0; i < npts; i++) {
        int64_t m = pm[i], n = pn[i];
        double cabs;
        double c = point_f64(dec, aq + m * lda, as, M, m, bq + n * ldb, bs + n, N, KB, &cabs);
        if (out_f64)
            out_f64[i] = c;
        if (out_abs)
            out_abs[i] = cabs;
        if (out_f32)
            out_f32[i] = point_f32(dec, aq + m * lda, as, M, m, bq + n * ldb, bs + n, N, KB);
    }
}

/* Grouped GEMM for routed experts: row r belongs to expert e with off[e] <= r < off[e+1]
 * and uses that expert's codes wq + e*N*ldw and scales ws + e*ceil(N/128)*(K/128).
 * aq [R][lda], as [K/128][R]. Selected elements (pr[i], pn[i]). */
void orc_grouped_gemm_points(const uint8_t *aq, int64_t lda, const float *as,
                             const uint8_t *wq, int64_t ldw, const float *ws,
                             const int32_t *off, int64_t G, int64_t R, int64_t N, int64_t K,
                             int64_t npts, const int64_t *pr, const int64_t *pn,
                             double *out_f64, double *out_abs)
{
    int64_t KB = K / 128;
    int64_t NB = (N + 127) / 128;
    double dec[256];
    dec_table(dec);
    for (int64_t i = 0; i < npts; i++) {
        int64_t r = pr[i], n = pn[i];
        int64_t e = 0;
        double cabs;
        double c;
        while (e < G && !(off[e] <= r && r < off[e + 1]))
            e++;
        if (e == G) {                     /* row outside every group: no defined value */
            if (out_f64)
                out_f64[i] = NAN;
            if (out_abs)
                out_abs[i] = NAN;
            continue;
        }
        c = point_f64(dec, aq + r * lda, as, R, r,
                      wq + (e * N + n) * ldw, ws + (e * NB + n / 128) * KB, 1, KB, &cabs);
        if (out_f64)
            out_f64[i] = c;
        if (out_abs)
            out_abs[i] = cabs;
    }
}

/* SwiGLU between the two expert GEMMs, h = silu(g) * u with silu(x) = x / (1 + e^-x), in FP64.
 * A reading: the pages name DeepSeekMoE's routed experts but not the activation between their
 * two GEMMs; DeepSeek-V3's expert FFN uses SwiGLU. For x below about -709, e^-x overflows to
 * +inf and silu(x) is -0. */
void orc_swiglu_f64(const double *g, const double *u, int64_t n, double *h)
{
    for (int64_t i = 0; i < n; i++)
        h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* MoE dispatch, token side ([MoE]: each token routed to 8 of 256 experts; the expert GEMMs run on
 * rows sorted by expert). Permute: row r of the sorted operand is token tok[r]'s row, codes and
 * 1x128 scales alike: qp[r][k] = q[tok[r]][k], sp[kb][r] = s[kb][tok[r]].
 * q [T][ldq], s [K/128][T]; qp [R][ldqp], sp [K/128][R]. */
void orc_moe_permute(const uint8_t *q, int64_t ldq, const float *s, int64_t T,
                     const int32_t *tok, int64_t R, int64_t K, uint8_t *qp, int64_t ldqp, float *sp)
{
    int64_t KB = K / 128;
    for (int64_t r = 0; r < R; r++) {
        int64_t t = tok[r];
        for (int64_t k = 0; k < K; k++)
            qp[r * ldqp + k] = q[t * ldq + k];
        for (int64_t kb = 0; kb < KB; kb++)
            sp[kb * R + r] = s[kb * T + t];
    }
}

/* MoE combine: token t's output is the routing-weighted sum of its expert rows,
 * out[t][n] = sum_j w[t][j] * y[row[t][j]][n], summed in FP32 as acc = fmaf(w, y, acc) for
 * j = 0 .. topk-1 in order from acc = 0, then rounded to BF16 (nearest, ties to even).
 * y BF16 bits [R][ldy]; row int32 [T][topk]; w FP32 [T][topk]; out BF16 bits [T][ldo]. */
void orc_moe_combine(const uint16_t *y, int64_t ldy, const int32_t *row, const float *w,
                     int64_t T, int64_t topk, int64_t N, uint16_t *out, int64_t ldo)
{
    for (int64_t t = 0; t < T; t++)
        for (int64_t n = 0; n < N; n++) {
            float acc = 0.0f;
            for (int64_t j = 0; j < topk; j++)
                acc = fmaf(w[t * topk + j], bf16_bits_to_float(y[(int64_t)row[t * topk + j] * ldy + n]),
                           acc);
            out[t * ldo + n] = float_to_bf16_rne(acc);
        }
}

/* Unquantized FP64 product of the BF16 inputs, C[m][n] = sum_k x[m,k] * w[n,k]; used only to
 * check the oracle itself against the quantization error bound. */
void orc_gemm_unquantized_f64(const uint16_t *x, int64_t ldx, const uint16_t *w, int64_t ldw,
                              int64_t M, int64_t N, int64_t K, double *c)
{
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; k++)
                acc += (double)bf16_bits_to_float(x[m * ldx + k]) *
                       (double)bf16_bits_to_float(w[n * ldw + k]);
            c[m * N + n] = acc;
        }
}
