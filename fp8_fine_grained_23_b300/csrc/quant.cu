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

#include "e4m3.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {

namespace {

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
// 1x128 activation tiles: one warp per run of QA_TILES consecutive tiles of one row.
//
// Half-warp h holds the tiles 2i + h (i < QA_TILES / 2) of the run; lane l16 of the half holds
// eight values (16 bytes) of each, so every load instruction of the warp reads 512 contiguous
// bytes of the row, and all of a warp's loads are issued before any is used (QA_TILES * 256
// bytes in flight per warp, six 8-warp CTAs per SM). A tile's amax is the packed 16-bit
// maximum of |bits| over the lane's eight values (exact for finite BF16), reduced over the 16
// lanes of its half by four xor shuffles, two tiles per 32-bit word. Lane l16 < QA_TILES / 2 then
// forms the scale of its half's tile 2 l16 + h (the two IEEE divisions run once per tile and are
// stored by that lane), and every lane receives r and the tile's mode by shuffles to encode its
// values; each store instruction writes 256 contiguous code bytes. No shared memory, no waits.
// ------------------------------------------------------------------------------------
constexpr int QA_TILES = 8;            // tiles per warp
constexpr int QA_WARPS = 8;            // warps per CTA
constexpr int QA_THREADS = QA_WARPS * 32;
constexpr int QA_CTAS_PER_SM = 6;      // 40 registers: 48 warps, 96 KB of loads in flight per SM

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// max |x| of eight BF16 values held as four 32-bit words, as BF16 bits: for finite BF16 the
// magnitude order is the unsigned order of the bits with the sign cleared.
__device__ __forceinline__ uint32_t absmax_bits8(const uint4& v)
{
    uint32_t m = max_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
    m = max_u16x2(m, v.z & 0x7FFF7FFFu);
    m = max_u16x2(m, v.w & 0x7FFF7FFFu);
    return max(m & 0xFFFFu, m >> 16);
}

template <bool UE8M0>
__global__ void __launch_bounds__(QA_THREADS, QA_CTAS_PER_SM)
quant_act_1x128_kernel(const uint16_t* __restrict__ x, int64_t M, int KB, int64_t ldx,
                       uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scales)
{
    constexpr int H = QA_TILES / 2;   // tiles per half-warp
    const int lane = threadIdx.x & 31, half = lane >> 4, l16 = lane & 15;
    const int runs = (KB + QA_TILES - 1) / QA_TILES;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * QA_WARPS + (threadIdx.x >> 5);
    if (wid >= M * runs) return;      // whole warps only
    const int64_t row = wid / runs;
    const int tile0 = static_cast<int>(wid % runs) * QA_TILES;
    const int nt = min(QA_TILES, KB - tile0);
    const uint16_t* src = x + row * ldx + static_cast<int64_t>(tile0) * 128 + l16 * 8;
    uint4 v[H];
#pragma unroll
    for (int i = 0; i < H; i++) {
        const int t = 2 * i + half;
        v[i] = t < nt ? ld_stream_v4(src + t * 128) : make_uint4(0u, 0u, 0u, 0u);
    }
    // P[k]: this half's tiles 4k + h (low 16 bits) and 4k + 2 + h (high 16 bits)
    uint32_t P[H / 2];
#pragma unroll
    for (int k = 0; k < H / 2; k++) P[k] = absmax_bits8(v[2 * k]) | (absmax_bits8(v[2 * k + 1]) << 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
#pragma unroll
        for (int k = 0; k < H / 2; k++) P[k] = max_u16x2(P[k], __shfl_xor_sync(0xffffffffu, P[k], o));
    }
    uint32_t mine = 0;   // amax bits of tile 2 * l16 + half (lanes l16 < H)
#pragma unroll
    for (int k = 0; k < H / 2; k++)
        if ((l16 >> 1) == k) mine = (l16 & 1) ? (P[k] >> 16) : (P[k] & 0xFFFFu);
    const TileScale ts = tile_scale_of<UE8M0>(__uint_as_float(mine << 16));
    const int my_tile = 2 * l16 + half;
    if (l16 < H && my_tile < nt) scales[static_cast<int64_t>(tile0 + my_tile) * M + row] = ts.s;
    const uint32_t mode = (ts.tiny ? 1u : 0u) | (ts.zero ? 2u : 0u);
    uint8_t* dst = q + row * ldq + static_cast<int64_t>(tile0) * 128 + l16 * 8;
#pragma unroll
    for (int i = 0; i < H; i++) {
        TileScale ti;
        ti.r = __shfl_sync(0xffffffffu, ts.r, (half << 4) + i);
        const uint32_t md = __shfl_sync(0xffffffffu, mode, (half << 4) + i);
        ti.tiny = (md & 1u) != 0;
        ti.zero = (md & 2u) != 0;
        const int t = 2 * i + half;
        float f[8];
        unpack_bf16x8(v[i], f);
        if (t < nt) st_v2(dst + t * 128, encode8(f, ti));
    }
}

// ------------------------------------------------------------------------------------
// 128x128 weight blocks: one CTA per block (blockIdx.x = K block, blockIdx.y = row block).
// Thread t reads 16 bytes of rows (t/16) + 16 i, i = 0..7, so the block is read from HBM once
// and held in registers while its amax is reduced (warp shuffles, then shared memory).
// ------------------------------------------------------------------------------------
// Four CTAs per SM (64 registers, a few spilled) keep 128 KB of loads in flight per SM: 95% of
// HBM against 91% at three (80 registers).
template <bool UE8M0>
__global__ void __launch_bounds__(QUANT_THREADS, 4)
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

    const TileScale ts = tile_scale_of<UE8M0>(a);
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

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, const uint2& v)
{
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_global_v4(void* p, const uint4& v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// ------------------------------------------------------------------------------------
// Backward-pass quantizers with transposed codes (the pages use E4M3 for the backward pass
// too: codingmall.com "Định dạng E4M3 hợp nhất", dtcms.com 三.2). A contraction over the rows
// of the input needs the codes with those rows contiguous, so both write qt[c][r].
//   PER_COLUMN (128x1 tiles): one scale per column of a 128x128 block, i.e. per 128 tokens of
//     one channel, for the weight-gradient GEMM; scales[rb * scale_ld + c] (c = global column).
//   else (128x128 blocks): one scale per block, the forward weight blocks laid out as W^T for
//     the data-gradient GEMM; scales[cb * scale_ld + rb].
// One CTA per 128x128 block (rb = blockIdx.y, cb = blockIdx.x). Thread t holds rows
// 8 * (t >> 4) .. + 7 and columns 8 * (t & 15) .. + 7 (eight coalesced 16-byte loads). The
// codes of one column are formed straight from the held values (eight rows -> eight bytes)
// and staged in a 128 x 128-byte tile whose 16-byte chunk j of row c sits at j ^ ((c >> 3) & 7),
// which keeps both the 8-byte writes and the 16-byte reads free of bank conflicts; the tile
// then leaves as 128 rows of 128 contiguous bytes.
// ------------------------------------------------------------------------------------
template <bool PER_COLUMN>
__global__ void __launch_bounds__(QUANT_THREADS)
quant_transpose_kernel(const uint16_t* __restrict__ x, int64_t ldx, uint8_t* __restrict__ qt,
                       int64_t ldqt, float* __restrict__ scales, int64_t scale_ld)
{
    __shared__ float red[QUANT_THREADS / 32][128];
    __shared__ float col_r[128];
    __shared__ uint32_t col_mode[128];   // bit 0: tiny amax, bit 1: zero tile
    __shared__ __align__(16) uint8_t tile[128 * 128];

    const int t = threadIdx.x;
    const int c8 = t & 15;
    const int rg = t >> 4;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; i++)
        v[i] = ld_stream_v4(x + (r0 + rg * 8 + i) * ldx + c0 + c8 * 8);

    // |x| maxima: per column of this thread (PER_COLUMN) or over everything it holds.
    float cm[8];
#pragma unroll
    for (int j = 0; j < 8; j++) cm[j] = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        float f[8];
        unpack_bf16x8(v[i], f);
#pragma unroll
        for (int j = 0; j < 8; j++) cm[j] = fmaxf(cm[j], fabsf(f[j]));
    }
    if constexpr (PER_COLUMN) {
        // lanes l and l ^ 16 hold the same columns (row groups 2w and 2w + 1)
#pragma unroll
        for (int j = 0; j < 8; j++) cm[j] = fmaxf(cm[j], __shfl_xor_sync(0xffffffffu, cm[j], 16));
        if (lane < 16) {
#pragma unroll
            for (int j = 0; j < 8; j++) red[warp][c8 * 8 + j] = cm[j];
        }
        __syncthreads();
        if (t < 128) {
            float a = red[0][t];
#pragma unroll
            for (int w = 1; w < QUANT_THREADS / 32; w++) a = fmaxf(a, red[w][t]);
            const TileScale ts = tile_scale(a);
            col_r[t] = ts.r;
            col_mode[t] = (ts.tiny ? 1u : 0u) | (ts.zero ? 2u : 0u);
            scales[static_cast<int64_t>(blockIdx.y) * scale_ld + c0 + t] = ts.s;
        }
    } else {
        float a = cm[0];
#pragma unroll
        for (int j = 1; j < 8; j++) a = fmaxf(a, cm[j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (lane == 0) red[warp][0] = a;
        __syncthreads();
        if (t == 0) {
            a = red[0][0];
#pragma unroll
            for (int w = 1; w < QUANT_THREADS / 32; w++) a = fmaxf(a, red[w][0]);
            const TileScale ts = tile_scale(a);
            col_r[0] = ts.r;
            col_mode[0] = (ts.tiny ? 1u : 0u) | (ts.zero ? 2u : 0u);
            scales[static_cast<int64_t>(blockIdx.x) * scale_ld + blockIdx.y] = ts.s;
        }
    }
    __syncthreads();

    // Column c8 * 8 + j, rows rg * 8 .. + 7 -> eight code bytes (row order), one 8-byte store.
    const uint32_t tile_base = smem_u32(tile);
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const int c = c8 * 8 + j;
        const float r = PER_COLUMN ? col_r[c] : col_r[0];
        const uint32_t mode = PER_COLUMN ? col_mode[c] : col_mode[0];
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t wd = (j & 2) ? ((j & 4) ? v[i].w : v[i].y) : ((j & 4) ? v[i].z : v[i].x);
            const float f = __uint_as_float((j & 1) ? (wd & 0xFFFF0000u) : (wd << 16));
            y[i] = (mode & 1u) ? __fmul_rn(__fmul_rn(f, 0x1p64f), r) : __fmul_rn(f, r);
        }
        uint32_t w0 = cvt_e4m3x2(y[0], y[1]) | (cvt_e4m3x2(y[2], y[3]) << 16);
        uint32_t w1 = cvt_e4m3x2(y[4], y[5]) | (cvt_e4m3x2(y[6], y[7]) << 16);
        if (mode & 2u) w0 = w1 = 0u;
        const uint32_t chunk = static_cast<uint32_t>((rg >> 1) ^ (c8 & 7));
        st_shared_v2(tile_base + c * 128 + chunk * 16 + (rg & 1) * 8, make_uint2(w0, w1));
    }
    __syncthreads();

    // 128 rows of 128 bytes: thread t writes chunks (t + 256 p), eight threads per row.
#pragma unroll
    for (int pass = 0; pass < 4; pass++) {
        const int idx = pass * QUANT_THREADS + t;
        const int c = idx >> 3;
        const int q = idx & 7;
        const uint4 val = ld_shared_v4(tile_base + c * 128 + ((q ^ ((c >> 3) & 7)) * 16));
        st_global_v4(qt + (c0 + c) * ldqt + r0 + q * 16, val);
    }
}

}  // namespace

cudaError_t launch_quant_act(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                             int64_t ldq, float* scales, bool ue8m0, cudaStream_t stream)
{
    const int KB = static_cast<int>(K / 128);
    const int64_t warps = M * ((KB + QA_TILES - 1) / QA_TILES);
    const int64_t grid = (warps + QA_WARPS - 1) / QA_WARPS;
    if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
    auto kern = ue8m0 ? quant_act_1x128_kernel<true> : quant_act_1x128_kernel<false>;
    kern<<<static_cast<unsigned>(grid), QA_THREADS, 0, stream>>>(static_cast<const uint16_t*>(x), M,
                                                                 KB, ldx, q, ldq, scales);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                int64_t ldq, float* scales, bool ue8m0, cudaStream_t stream)
{
    const int KB = static_cast<int>(K / 128);
    const int64_t NB = (N + 127) / 128;
    dim3 grid(KB, static_cast<unsigned>(NB));
    auto kern = ue8m0 ? quant_weight_128x128_kernel<true> : quant_weight_128x128_kernel<false>;
    kern<<<grid, QUANT_THREADS, 0, stream>>>(static_cast<const uint16_t*>(w), N, KB, ldw, q, ldq,
                                             scales);
    return cudaGetLastError();
}

cudaError_t launch_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* qt,
                                   int64_t ldqt, float* scales, cudaStream_t stream)
{
    dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(M / 128));
    quant_transpose_kernel<true><<<grid, QUANT_THREADS, 0, stream>>>(
        static_cast<const uint16_t*>(x), ldx, qt, ldqt, scales, K);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight_t(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* qt,
                                  int64_t ldqt, float* scales_t, cudaStream_t stream)
{
    dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(N / 128));
    quant_transpose_kernel<false><<<grid, QUANT_THREADS, 0, stream>>>(
        static_cast<const uint16_t*>(w), ldw, qt, ldqt, scales_t, N / 128);
    return cudaGetLastError();
}

}  // namespace fp8bs
