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
// 1x128 activation tiles: persistent CTAs, TMA-staged, one tile per lane.
//
// The rows are cut into segments of up to 32 tiles (8 KB of BF16) of one row; each CTA owns a
// contiguous, balanced range of segments. Segment i of a CTA belongs to consumer warp i % QA_CONSUMERS,
// which owns QA_SLOTS_PER_WARP shared-memory slots and consumes them strictly in order (so every
// slot's mbarriers see one producer and one consumer, phase after phase). A producer thread
// streams the segments, in order, into the slots with bulk copies (QA_SLOTS x 8 KB in flight
// per CTA). A consumer warp takes a whole segment: lane l loads tile l (16 x 16 B, rotated so that the reads are free of
// bank conflicts), reduces its amax with packed 16-bit integer maxima on |bits| (exact for
// finite BF16), computes its scale and reciprocal (one division pass covers 32 tiles), and
// encodes its 128 values. The codes are written back into the slot and then copied out with
// coalesced 16-byte stores (512 contiguous bytes per warp instruction).
// ------------------------------------------------------------------------------------
constexpr int SEG_TILES = 32;
constexpr int SEG_BYTES = SEG_TILES * 256;
constexpr int QA_CONSUMERS = 6;
constexpr int QA_SLOTS_PER_WARP = 2;
constexpr int QA_SLOTS = QA_CONSUMERS * QA_SLOTS_PER_WARP;
constexpr int QA_THREADS = (QA_CONSUMERS + 1) * 32;
constexpr int QA_CTAS_PER_SM = 2;
constexpr int QA_SMEM = QA_SLOTS * SEG_BYTES + 2 * QA_SLOTS * 8 + 16 + 128;

struct QuantActArgs {
    const uint16_t* x;
    int64_t M;
    int KB;
    int64_t ldx;
    uint8_t* q;
    int64_t ldq;
    float* scales;
    int* err;
    long long budget;
};

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

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// max |x| over eight BF16 values held as four 32-bit words: for finite BF16 the magnitude order
// is the unsigned order of the bits with the sign cleared.
__device__ __forceinline__ uint32_t absmax_bits_u16x2(const uint4& v, uint32_t m)
{
    m = max_u16x2(m, v.x & 0x7FFF7FFFu);
    m = max_u16x2(m, v.y & 0x7FFF7FFFu);
    m = max_u16x2(m, v.z & 0x7FFF7FFFu);
    return max_u16x2(m, v.w & 0x7FFF7FFFu);
}

// Slot and barrier phase of a CTA's i-th segment: consumer warp w = i % QA_CONSUMERS handles
// its k-th segment (k = i / QA_CONSUMERS) in its own slot w * QA_SLOTS_PER_WARP +
// k % QA_SLOTS_PER_WARP, which it has used k / QA_SLOTS_PER_WARP times before.
__device__ __forceinline__ uint32_t qa_slot(int64_t i)
{
    const int64_t w = i % QA_CONSUMERS, k = i / QA_CONSUMERS;
    return static_cast<uint32_t>(w * QA_SLOTS_PER_WARP + k % QA_SLOTS_PER_WARP);
}

__device__ __forceinline__ uint32_t qa_phase(int64_t i)
{
    return static_cast<uint32_t>((i / QA_CONSUMERS) / QA_SLOTS_PER_WARP) & 1u;
}

template <bool UE8M0>
__global__ void __launch_bounds__(QA_THREADS, QA_CTAS_PER_SM)
quant_act_1x128_kernel(const QuantActArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    const uint32_t bar_full = base + QA_SLOTS * SEG_BYTES;
    const uint32_t bar_empty = bar_full + 8 * QA_SLOTS;
    const uint32_t abort_addr = bar_empty + 8 * QA_SLOTS;   // shared word: a role gave up

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int KB = p.KB;
    const int segs_per_row = (KB + SEG_TILES - 1) / SEG_TILES;
    const int64_t total = p.M * segs_per_row;
    const int64_t s_begin = total * blockIdx.x / gridDim.x;
    const int64_t nseg = total * (blockIdx.x + 1) / gridDim.x - s_begin;

    if (threadIdx.x == 0) {
        for (int i = 0; i < QA_SLOTS; i++) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, 1);
        }
        st_shared_volatile_u32(abort_addr, 0u);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == QA_CONSUMERS) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int64_t i = 0;
            bool ok = true;
            for (; i < nseg; i++) {
                const uint32_t slot = qa_slot(i);
                const uint32_t ph = qa_phase(i);
                if (!mbar_wait(bar_empty + 8 * slot, ph ^ 1u, abort_addr, p.budget)) {
                    st_shared_volatile_u32(abort_addr, 1u);
                    atomicCAS(p.err, 0, DEV_TIMEOUT_PRODUCER);
                    ok = false;
                    break;
                }
                const int64_t seg = s_begin + i;
                const int64_t row = seg / segs_per_row;
                const int tile0 = static_cast<int>(seg % segs_per_row) * SEG_TILES;
                const int nt = min(SEG_TILES, KB - tile0);
                const uint32_t bytes = static_cast<uint32_t>(nt) * 256u;
                mbar_arrive_expect_tx(bar_full + 8 * slot, bytes);
                bulk_load(base + slot * SEG_BYTES, p.x + row * p.ldx + static_cast<int64_t>(tile0) * 128,
                          bytes, bar_full + 8 * slot);
            }
            if (!ok || ld_shared_volatile_u32(abort_addr) != 0) {
                // after an abort, wait for the copies already issued before the CTA exits
                for (int64_t j = (i > QA_SLOTS ? i - QA_SLOTS : 0); j < i; j++)
                    if (!mbar_wait(bar_full + 8 * qa_slot(j), qa_phase(j), 0u, p.budget))
                        atomicCAS(p.err, 0, DEV_TIMEOUT_DRAIN);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        for (int64_t i = warp; i < nseg; i += QA_CONSUMERS) {
            const uint32_t slot = qa_slot(i);
            const uint32_t ph = qa_phase(i);
            const bool got = mbar_wait(bar_full + 8 * slot, ph, abort_addr, p.budget);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) {
                    st_shared_volatile_u32(abort_addr, 1u);
                    atomicCAS(p.err, 0, DEV_TIMEOUT_EPILOGUE);
                }
                break;
            }
            const int64_t seg = s_begin + i;
            const int64_t row = seg / segs_per_row;
            const int tile0 = static_cast<int>(seg % segs_per_row) * SEG_TILES;
            const int nt = min(SEG_TILES, KB - tile0);
            const bool active = lane < nt;
            const uint32_t slot_base = base + slot * SEG_BYTES;
            const uint32_t my_tile = slot_base + lane * 256;

            uint4 v[16];
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const int c = (j + lane) & 15;
                v[j] = active ? ld_shared_v4(my_tile + c * 16) : make_uint4(0u, 0u, 0u, 0u);
            }
            uint32_t m2 = 0;
#pragma unroll
            for (int j = 0; j < 16; j++) m2 = absmax_bits_u16x2(v[j], m2);
            const uint32_t mbits = max(m2 & 0xFFFFu, m2 >> 16);
            const TileScale ts = tile_scale_of<UE8M0>(__uint_as_float(mbits << 16));
            __syncwarp();   // every lane holds its tile before the codes overwrite the slot

#pragma unroll
            for (int j = 0; j < 16; j++) {
                const int c = (j + lane) & 15;
                float f[8];
                unpack_bf16x8(v[j], f);
                const uint2 codes = encode8(f, ts);
                if (active) st_shared_v2(slot_base + lane * 128 + c * 8, codes);
            }
            __syncwarp();

            const int code_bytes = nt * 128;
            uint8_t* qrow = p.q + row * p.ldq + static_cast<int64_t>(tile0) * 128;
#pragma unroll
            for (int j = 0; j < SEG_TILES * 128 / 512; j++) {
                const int off = j * 512 + lane * 16;
                if (off < code_bytes) st_global_v4(qrow + off, ld_shared_v4(slot_base + off));
            }
            if (active) p.scales[static_cast<int64_t>(tile0 + lane) * p.M + row] = ts.s;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
        }
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
                             int64_t ldq, float* scales, int num_sms, int* err, long long budget,
                             bool ue8m0, cudaStream_t stream)
{
    QuantActArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.M = M;
    a.KB = static_cast<int>(K / 128);
    a.ldx = ldx;
    a.q = q;
    a.ldq = ldq;
    a.scales = scales;
    a.err = err;
    a.budget = budget;
    const int64_t segs = M * ((a.KB + SEG_TILES - 1) / SEG_TILES);
    const int64_t cap = static_cast<int64_t>(num_sms) * QA_CTAS_PER_SM;
    const int grid = static_cast<int>(segs < cap ? segs : cap);
    auto kern = ue8m0 ? quant_act_1x128_kernel<true> : quant_act_1x128_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, QA_SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, QA_THREADS, QA_SMEM, stream>>>(a);
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
