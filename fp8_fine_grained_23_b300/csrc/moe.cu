// moe.cu -- MoE dispatch on the token side: permute token rows (FP8 codes and their 1x128
// scales) into the expert-sorted order the grouped GEMMs read, and combine each token's expert
// outputs with its routing weights.
//
// The pages route each token to 8 of 256 routed experts (dtcms.com 一.2 "DeepSeekMoE架构",
// risenshineclean.com 二); the grouped GEMM runs on rows sorted by expert. Both kernels are
// HBM-bound gathers: permute moves 2 bytes per code element (read + write) plus the scales;
// combine reads topk BF16 rows per token and writes one.
#include <cstdint>

#include "internal.h"

namespace fp8bs {

namespace {

constexpr int MOE_THREADS = 256;
constexpr int MOE_WARPS = MOE_THREADS / 32;

__device__ __forceinline__ uint4 ld_nc_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4_global(void* p, const uint4& v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Warp w of block b copies sorted row r = 8 b + w: qp[r] = q[tok[r]] (K bytes, 16 per lane per
// step); then the block writes its 8 rows' scales, sp[kb][r] = s[kb][tok[r]] (8 consecutive
// floats per K block). A token index outside [0, T) is outside the contract: its row is not
// written.
__global__ void __launch_bounds__(MOE_THREADS)
moe_permute_kernel(const uint8_t* __restrict__ q, int64_t ldq, const float* __restrict__ s,
                   int64_t T, const int32_t* __restrict__ tok, int64_t R, int K,
                   uint8_t* __restrict__ qp, int64_t ldqp, float* __restrict__ sp)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * MOE_WARPS + warp;
    if (r < R) {
        const int64_t t = tok[r];
        if (t >= 0 && t < T) {
            const uint8_t* src = q + t * ldq;
            uint8_t* dst = qp + r * ldqp;
            for (int i = lane; i < K / 16; i += 32) st_v4_global(dst + 16 * i, ld_nc_v4(src + 16 * i));
        }
    }
    const int KB = K / 128;
    for (int idx = threadIdx.x; idx < MOE_WARPS * KB; idx += MOE_THREADS) {
        const int kb = idx / MOE_WARPS;
        const int64_t rr = static_cast<int64_t>(blockIdx.x) * MOE_WARPS + idx % MOE_WARPS;
        if (rr >= R) continue;
        const int64_t t = tok[rr];
        if (t >= 0 && t < T) sp[kb * R + rr] = s[kb * T + t];
    }
}

// Token t = one warp: out[t][n] = sum_j w[t][j] * y[row[t][j]][n] as an FP32 fma chain in
// j order from 0, rounded to BF16 (nearest even).
// A row index outside [0, R) adds nothing (outside the contract).
__global__ void __launch_bounds__(MOE_THREADS)
moe_combine_kernel(const uint16_t* __restrict__ y, int64_t ldy, int64_t R,
                   const int32_t* __restrict__ row, const float* __restrict__ w, int64_t T,
                   int topk, int N, uint16_t* __restrict__ out, int64_t ldo)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * MOE_WARPS + (threadIdx.x >> 5);
    if (t >= T) return;
    // this token's rows and weights, one per lane (topk <= 32)
    int64_t my_row = -1;
    float my_w = 0.0f;
    if (lane < topk) {
        const int64_t rv = row[t * topk + lane];
        my_row = (rv >= 0 && rv < R) ? rv : -1;
        my_w = w[t * topk + lane];
    }
    // A warp step covers 2 KB of every row it reads (lane l: 16-byte chunks l, l + 32, l + 64,
    // l + 96 of the step, so that each load instruction reads 512 contiguous bytes), and the
    // gathered rows reach DRAM in long runs; rows go 4 at a time, their loads issued before their
    // fma chains.
    const int chunks = N / 8;
    for (int c0 = 0; c0 < chunks; c0 += 128) {
        float acc[4][8];
#pragma unroll
        for (int q = 0; q < 4; q++)
#pragma unroll
            for (int e = 0; e < 8; e++) acc[q][e] = 0.0f;
        for (int j0 = 0; j0 < topk; j0 += 4) {
            uint4 v[4][4];
            float wj[4];
#pragma unroll
            for (int jj = 0; jj < 4; jj++) {
                const int j = j0 + jj;
                const int64_t rj = __shfl_sync(0xffffffffu, my_row, j & 31);
                const bool use = j < topk && rj >= 0;
                wj[jj] = use ? __shfl_sync(0xffffffffu, my_w, j & 31) : 0.0f;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int c = c0 + lane + 32 * q;
                    v[jj][q] = (use && c < chunks) ? ld_nc_v4(y + rj * ldy + 8 * c)
                                                   : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int jj = 0; jj < 4; jj++) {
                if (j0 + jj >= topk) break;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const uint32_t wd[4] = {v[jj][q].x, v[jj][q].y, v[jj][q].z, v[jj][q].w};
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        acc[q][2 * e] =
                            __fmaf_rn(wj[jj], __uint_as_float(wd[e] << 16), acc[q][2 * e]);
                        acc[q][2 * e + 1] = __fmaf_rn(wj[jj], __uint_as_float(wd[e] & 0xFFFF0000u),
                                                      acc[q][2 * e + 1]);
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int c = c0 + lane + 32 * q;
            if (c >= chunks) continue;
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                uint32_t packed;
                asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
                    : "=r"(packed)
                    : "f"(acc[q][2 * e + 1]), "f"(acc[q][2 * e]));
                o[e] = packed;
            }
            st_v4_global(out + t * ldo + 8 * c, make_uint4(o[0], o[1], o[2], o[3]));
        }
    }
}

}  // namespace

cudaError_t launch_moe_permute(const uint8_t* q, int64_t ldq, const float* s, int64_t T,
                               const int32_t* tok, int64_t R, int64_t K, uint8_t* qp,
                               int64_t ldqp, float* sp, cudaStream_t stream)
{
    const int64_t blocks = (R + MOE_WARPS - 1) / MOE_WARPS;
    moe_permute_kernel<<<static_cast<unsigned>(blocks), MOE_THREADS, 0, stream>>>(
        q, ldq, s, T, tok, R, static_cast<int>(K), qp, ldqp, sp);
    return cudaGetLastError();
}

cudaError_t launch_moe_combine(const void* y, int64_t ldy, int64_t R, const int32_t* row,
                               const float* w, int64_t T, int64_t topk, int64_t N, void* out,
                               int64_t ldo, cudaStream_t stream)
{
    const int64_t blocks = (T + MOE_WARPS - 1) / MOE_WARPS;
    moe_combine_kernel<<<static_cast<unsigned>(blocks), MOE_THREADS, 0, stream>>>(
        static_cast<const uint16_t*>(y), ldy, R, row, w, T, static_cast<int>(topk),
        static_cast<int>(N), static_cast<uint16_t*>(out), ldo);
    return cudaGetLastError();
}

}  // namespace fp8bs
