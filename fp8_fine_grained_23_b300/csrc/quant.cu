// quant.cu -- online fine-grained E4M3 quantizers (1x128 activation tiles, 128x128 weight
// blocks), one FP32 scale per tile from the tile's own amax.
//
// Follows codingmall.com "Bạn có thể giải thích vai trò của độ chính xác FP8 trong quá trình
// đào tạo của DeepSeek-V3", sections "Định lượng hạt mịn" (1x128 tiles / 128x128 blocks, each
// scaled on its own) and "Định lượng trực tuyến" (scale from the current maximum), and
// risenshineclean.com section 三 (a 1x128 tile is one token by 128 channels).
//
// Both kernels are HBM-bound (2 bytes read, 1 + 4/128 bytes written per element for
// activations). Arithmetic per tile: FP32 max (exact), two IEEE FP32 divisions
// (s = amax/448, r = 448/amax), one FP32 multiply and one saturating round-to-nearest-even
// E4M3 conversion per element. Compiled without fast-math so that divisions are correctly
// rounded and subnormals are kept, which the bit-exact contract depends on.
#include <cstdint>

#include "internal.h"

namespace fp8bs {

namespace {

struct TileScale {
    float s;     // dequantization scale
    float r;     // quantization multiplier
    bool tiny;   // amax < 2^-64: r formed from amax * 2^64 (exact), values scaled by 2^64
    bool zero;   // amax == 0: scale 1, codes 0x00
};

__device__ __forceinline__ TileScale tile_scale(float amax)
{
    TileScale t;
    t.zero = (amax == 0.0f);
    t.tiny = !t.zero && (amax < 0x1p-64f);
    const float den = t.tiny ? __fmul_rn(amax, 0x1p64f) : amax;
    t.s = t.zero ? 1.0f : __fdiv_rn(amax, 448.0f);
    t.r = t.zero ? 0.0f : __fdiv_rn(448.0f, den);
    return t;
}

// Two FP32 values to two E4M3 codes, saturating round-to-nearest-even; `lo` lands in the low
// byte of the result.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ float absmax8(const float (&f)[8])
{
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) a = fmaxf(a, fabsf(f[i]));
    return a;
}

// Eight values of one tile to eight codes (byte i of the result is value i).
__device__ __forceinline__ uint2 encode8(const float (&f)[8], const TileScale& t)
{
    float y[8];
    if (t.tiny) {
#pragma unroll
        for (int i = 0; i < 8; i++) y[i] = __fmul_rn(__fmul_rn(f[i], 0x1p64f), t.r);
    } else {
#pragma unroll
        for (int i = 0; i < 8; i++) y[i] = __fmul_rn(f[i], t.r);
    }
    uint32_t w0 = cvt_e4m3x2(y[0], y[1]) | (cvt_e4m3x2(y[2], y[3]) << 16);
    uint32_t w1 = cvt_e4m3x2(y[4], y[5]) | (cvt_e4m3x2(y[6], y[7]) << 16);
    if (t.zero) w0 = w1 = 0u;
    return make_uint2(w0, w1);
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v2(void* p, const uint2& v)
{
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ------------------------------------------------------------------------------------
// 1x128 activation tiles.
// A half-warp (16 lanes x 8 BF16 = 128 values) owns one tile; each half-warp task covers
// TILES_PER_TASK consecutive tiles of one row, so a lane keeps that many 16-byte loads in
// flight. Tasks are numbered row-major, so a warp reads 2 x TILES_PER_TASK x 256 contiguous
// bytes. The loop runs per warp so that every shuffle sees all 32 lanes.
// ------------------------------------------------------------------------------------
constexpr int TILES_PER_TASK = 4;

__global__ void __launch_bounds__(QUANT_THREADS)
quant_act_1x128_kernel(const uint16_t* __restrict__ x, int64_t M, int KB, int64_t ldx,
                       uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scales)
{
    const int n_task_per_row = (KB + TILES_PER_TASK - 1) / TILES_PER_TASK;
    const int64_t T = M * n_task_per_row;
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;
    const int hl = lane & 15;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

    for (int64_t tw = warp0; 2 * tw < T; tw += nwarps) {
        const int64_t t = 2 * tw + half;
        const bool tv = t < T;
        const int64_t m = tv ? t / n_task_per_row : 0;
        const int kb0 = tv ? static_cast<int>(t % n_task_per_row) * TILES_PER_TASK : 0;

        uint4 v[TILES_PER_TASK];
#pragma unroll
        for (int i = 0; i < TILES_PER_TASK; i++) {
            const bool ok = tv && (kb0 + i < KB);
            v[i] = ok ? ld_stream_v4(x + m * ldx + static_cast<int64_t>(kb0 + i) * 128 + hl * 8)
                      : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < TILES_PER_TASK; i++) {
            const bool ok = tv && (kb0 + i < KB);
            float f[8];
            unpack_bf16x8(v[i], f);
            float a = absmax8(f);
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            const TileScale ts = tile_scale(a);
            const uint2 codes = encode8(f, ts);
            if (ok) {
                st_v2(q + m * ldq + static_cast<int64_t>(kb0 + i) * 128 + hl * 8, codes);
                if (hl == 0) scales[static_cast<int64_t>(kb0 + i) * M + m] = ts.s;
            }
        }
    }
}

// ------------------------------------------------------------------------------------
// 128x128 weight blocks: one CTA per block (blockIdx.x = K block, blockIdx.y = row block).
// Thread t reads 16 bytes of rows (t/16) + 16 i, i = 0..7, so the block is read from HBM once
// and held in registers while its amax is reduced (warp shuffles, then shared memory).
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(QUANT_THREADS)
quant_weight_128x128_kernel(const uint16_t* __restrict__ w, int64_t N, int KB, int64_t ldw,
                            uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scales)
{
    __shared__ float red[QUANT_THREADS / 32];
    const int kb = blockIdx.x;
    const int64_t nb = blockIdx.y;
    const int c8 = threadIdx.x & 15;
    const int r0 = threadIdx.x >> 4;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int64_t row = nb * 128 + r0 + 16 * i;
        v[i] = (row < N) ? ld_stream_v4(w + row * ldw + static_cast<int64_t>(kb) * 128 + c8 * 8)
                         : make_uint4(0u, 0u, 0u, 0u);
    }
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        float f[8];
        unpack_bf16x8(v[i], f);
        a = fmaxf(a, absmax8(f));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) red[warp] = a;
    __syncthreads();
    a = red[0];
#pragma unroll
    for (int i = 1; i < QUANT_THREADS / 32; i++) a = fmaxf(a, red[i]);

    const TileScale ts = tile_scale(a);
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int64_t row = nb * 128 + r0 + 16 * i;
        if (row < N) {
            float f[8];
            unpack_bf16x8(v[i], f);
            st_v2(q + row * ldq + static_cast<int64_t>(kb) * 128 + c8 * 8, encode8(f, ts));
        }
    }
    if (threadIdx.x == 0) scales[nb * KB + kb] = ts.s;
}

}  // namespace

cudaError_t launch_quant_act(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                             int64_t ldq, float* scales, int num_sms, cudaStream_t stream)
{
    const int KB = static_cast<int>(K / 128);
    const int64_t tasks = M * ((KB + TILES_PER_TASK - 1) / TILES_PER_TASK);
    const int64_t warps = (tasks + 1) / 2;
    const int64_t want = (warps + QUANT_THREADS / 32 - 1) / (QUANT_THREADS / 32);
    const int64_t cap = static_cast<int64_t>(num_sms) * (2048 / QUANT_THREADS);
    const int grid = static_cast<int>(want < cap ? want : cap);
    quant_act_1x128_kernel<<<grid, QUANT_THREADS, 0, stream>>>(
        static_cast<const uint16_t*>(x), M, KB, ldx, q, ldq, scales);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                int64_t ldq, float* scales, cudaStream_t stream)
{
    const int KB = static_cast<int>(K / 128);
    const int64_t NB = (N + 127) / 128;
    dim3 grid(KB, static_cast<unsigned>(NB));
    quant_weight_128x128_kernel<<<grid, QUANT_THREADS, 0, stream>>>(
        static_cast<const uint16_t*>(w), N, KB, ldw, q, ldq, scales);
    return cudaGetLastError();
}

}  // namespace fp8bs
