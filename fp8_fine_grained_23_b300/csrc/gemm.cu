// gemm.cu -- block-scaled FP8 GEMM (dense and grouped over routed experts) for sm_103a.
//
// What it computes (dtcms.com DeepSeek-V3 overview, section 三.1 and 三.3; codingmall.com
// "Tăng độ chính xác tích lũy"): C = A W^T from E4M3 operands, where every 128-wide K block
// carries its own scales (one per 1x128 activation tile, one per 128x128 weight block). The
// partial sum of each K block is formed by the tensor cores in FP32 and then promoted: it is
// multiplied by s_a[m] * s_w[n/128] and added to an FP32 accumulator. The pages do this on
// Hopper by copying WGMMA partials to CUDA-core registers at intervals; here the interval is one
// quantization block and the partial lives in tensor memory (TMEM) until the epilogue warps
// drain it, which overlaps with the MMAs of the next K block.
//
// Structure of one persistent CTA (384 threads = 3 warpgroups, one CTA per SM):
//   warp 0     TMA producer: streams 128x128 A and 256x128 W code tiles into a STAGES-deep
//              shared-memory ring (128-byte swizzle), completion tracked by mbarriers;
//   warp 1     TMEM owner and MMA issuer: for each K block, four tcgen05.mma (K = 32 each,
//              kind::f8f6f4, E4M3 x E4M3 -> FP32) into one of two 128x256 TMEM accumulators,
//              then tcgen05.commit to free the smem stage and to hand the partial to the
//              epilogue;
//   warps 2-3  idle after set-up (warp 0 also builds the group table of the grouped variant);
//   warps 4-11 epilogue: warp w reads TMEM lanes 32*(w%4).. (its rows) and columns
//              128*((w-4)/4).. (one weight block), promotes each K block's partial into 128
//              FP32 registers per thread, and writes the finished tile (BF16 or FP32).
// Registers: the launch gives 168 per thread (65536 / 384, rounded to 8). Warpgroup 0 drops to
// 56 and the two epilogue warpgroups rise to 224 (128*56 + 256*224 = 384*168), which holds the
// 128 accumulators and 64 staging registers of a thread without spilling.
// Every mbarrier wait is bounded (clock budget); on expiry the CTA records an error code in the
// device error word, stops issuing work, waits for its in-flight copies and MMAs, frees TMEM and
// returns.
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {

namespace {

constexpr int BM = GEMM_BM;
constexpr int BN = GEMM_BN;
constexpr int BK = GEMM_BK;
constexpr int STAGES = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int PRODUCER_WARP = 0;
constexpr int MMA_WARP = 1;
constexpr int EPI_WARP0 = 4;
constexpr int THREADS = 384;
constexpr int REGS_CONTROL = 56;           // warpgroup 0 after setmaxnreg.dec
constexpr int REGS_EPILOGUE = 224;         // warpgroups 1 and 2 after setmaxnreg.inc
static_assert(128 * REGS_CONTROL + 256 * REGS_EPILOGUE == THREADS * 168,
              "register split must equal the launch allocation of 168 per thread");
constexpr int TMEM_COLS = 2 * BN;          // two FP32 accumulators of 128 lanes x BN columns

constexpr int A_BYTES = BM * BK;           // E4M3: one byte per element
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int A_OFF = 0;
constexpr int B_OFF = STAGES * A_BYTES;
constexpr int BAR_OFF = STAGES * STAGE_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 5;   // full[S], empty[S], tfull[2], tempty[2], drain
constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
constexpr int GROUP_OFF = MISC_OFF + 16;
constexpr int ALIGN_PAD = 1024;            // 128-byte-swizzled tiles need 1024-byte alignment

static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "tiles must keep 1024-B alignment");

struct TileInfo {
    int64_t row0;      // first row of the tile in A / C
    int64_t row_end;   // rows >= row_end are not stored (next group or past the end)
    int64_t wrow0;     // first row of the W code tile (group * N + n0)
    int n0;            // first output column
    int g;             // group (0 for dense)
};

__device__ __forceinline__ void raise_error(int* err, volatile int* abort_flag, int code)
{
    *abort_flag = 1;
    atomicCAS(err, 0, code);
}

template <bool GROUPED>
__device__ __forceinline__ TileInfo decode_tile(int t, const GemmArgs& p, const int* s_tstart,
                                                const int* s_off)
{
    TileInfo ti;
    if constexpr (!GROUPED) {
        const int mt = t % p.MT;
        const int nt = t / p.MT;
        ti.row0 = static_cast<int64_t>(mt) * BM;
        ti.row_end = p.rows;
        ti.n0 = nt * BN;
        ti.wrow0 = ti.n0;
        ti.g = 0;
    } else {
        // s_tstart[g] = first tile of group g; binary search for the last g with start <= t.
        int lo = 0, hi = p.G;   // invariant: s_tstart[lo] <= t < s_tstart[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_tstart[mid] <= t) lo = mid; else hi = mid;
        }
        const int g = lo;
        const int local = t - s_tstart[g];
        const int rows_g = s_off[g + 1] - s_off[g];
        const int mtg = (rows_g + BM - 1) / BM;
        const int nt = local / mtg;         // m-tiles of one (group, n-tile) are adjacent
        const int mt = local % mtg;
        ti.row0 = static_cast<int64_t>(s_off[g]) + static_cast<int64_t>(mt) * BM;
        const int64_t end = s_off[g + 1];
        ti.row_end = end < p.rows ? end : p.rows;
        ti.n0 = nt * BN;
        ti.wrow0 = static_cast<int64_t>(g) * p.N + ti.n0;
        ti.g = g;
    }
    return ti;
}

template <int N>
__device__ __forceinline__ void regs_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void regs_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void st_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

template <bool GROUPED, bool OUT_F32>
__global__ void __launch_bounds__(THREADS, 1)
fp8_blockscaled_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                            const __grid_constant__ CUtensorMap map_b, const GemmArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + (ALIGN_PAD - 1)) & ~static_cast<uint32_t>(ALIGN_PAD - 1);
    uint8_t* smem = smem_raw + (base - raw);

    const uint32_t sA = base + A_OFF;
    const uint32_t sB = base + B_OFF;
    const uint32_t bar0 = base + BAR_OFF;
    const uint32_t full0 = bar0;
    const uint32_t empty0 = bar0 + 8 * STAGES;
    const uint32_t tfull0 = bar0 + 16 * STAGES;
    const uint32_t tempty0 = tfull0 + 16;
    const uint32_t drain_bar = tempty0 + 16;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + MISC_OFF + 4);
    int* s_tstart = reinterpret_cast<int*>(smem + GROUP_OFF);   // grouped: [G+1]
    int* s_off = s_tstart + (p.G + 1);                            // grouped: [G+1]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long budget = p.budget;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, NUM_EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
        tmem_relinquish();
    }
    if constexpr (GROUPED) {
        // Group table: copy the offsets, then s_tstart[g] = sum over g' < g of
        // ceil(rows_g' / 128) * NT (an exclusive scan done by warp 0, 32 groups per step).
        if (warp == 0) {
            for (int g = lane; g <= p.G; g += 32) s_off[g] = __ldg(p.offsets + g);
            __syncwarp();
            int carry = 0;
            for (int g0 = 0; g0 < p.G; g0 += 32) {
                const int g = g0 + lane;
                int rows_g = (g < p.G) ? (s_off[g + 1] - s_off[g]) : 0;
                rows_g = rows_g > 0 ? rows_g : 0;
                const int v = ((rows_g + BM - 1) / BM) * p.NT;
                int incl = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                if (g < p.G) s_tstart[g] = carry + incl - v;
                carry += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) s_tstart[p.G] = carry;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    int num_tiles = p.num_tiles;
    if constexpr (GROUPED) num_tiles = s_tstart[p.G];
    const int KB = p.KB;

    if (warp < EPI_WARP0) {
        regs_dec<REGS_CONTROL>();
        if (warp == PRODUCER_WARP) {
            // ---------------------------------------------------------------- TMA producer
            if (lane == 0) {
                uint32_t it = 0;
                bool ok = true;
                for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
                    const TileInfo ti = decode_tile<GROUPED>(t, p, s_tstart, s_off);
                    for (int kb = 0; kb < KB; kb++, it++) {
                        const uint32_t s = it % STAGES;
                        const uint32_t ph = (it / STAGES) & 1u;
                        if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag, budget)) {
                            raise_error(p.err, abort_flag, DEV_TIMEOUT_PRODUCER);
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full0 + 8 * s, STAGE_BYTES);
                        tma_load_2d(sA + s * A_BYTES, &map_a, full0 + 8 * s, kb * BK,
                                    static_cast<int32_t>(ti.row0));
                        tma_load_2d(sB + s * B_BYTES, &map_b, full0 + 8 * s, kb * BK,
                                    static_cast<int32_t>(ti.wrow0));
                    }
                }
                if (!ok) {
                    // The MMA side may never consume what is in flight: wait for the last copy
                    // issued into every stage before the CTA may exit.
                    const uint32_t first = it > STAGES ? it - STAGES : 0;
                    for (uint32_t i = first; i < it; i++)
                        if (!mbar_wait(full0 + 8 * (i % STAGES), (i / STAGES) & 1u, nullptr, budget))
                            atomicCAS(p.err, 0, DEV_TIMEOUT_DRAIN);
                }
            }
        } else if (warp == MMA_WARP) {
            // ---------------------------------------------------------------- MMA issuer
            if (lane == 0) {
                constexpr uint32_t IDESC = idesc_e4m3_f32(BM, BN);
                uint32_t it = 0, j = 0;
                bool ok = true, issued = false;
                for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
                    for (int kb = 0; kb < KB; kb++, it++, j++) {
                        const uint32_t b = j & 1u;
                        const uint32_t pb = (j >> 1) & 1u;
                        if (!mbar_wait(tempty0 + 8 * b, pb ^ 1u, abort_flag, budget)) {
                            raise_error(p.err, abort_flag, DEV_TIMEOUT_MMA_TMEM);
                            ok = false;
                            break;
                        }
                        const uint32_t s = it % STAGES;
                        const uint32_t ph = (it / STAGES) & 1u;
                        if (!mbar_wait(full0 + 8 * s, ph, abort_flag, budget)) {
                            raise_error(p.err, abort_flag, DEV_TIMEOUT_MMA_FULL);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t da = desc_kmajor_sw128(sA + s * A_BYTES);
                        const uint64_t db = desc_kmajor_sw128(sB + s * B_BYTES);
                        const uint32_t d_tmem = tmem_base + b * BN;
    #pragma unroll
                        for (int k = 0; k < BK / 32; k++)   // +32 bytes of K = +2 in the address field
                            mma_e4m3(d_tmem, da + 2 * k, db + 2 * k, IDESC, k > 0 ? 1u : 0u);
                        mma_commit(empty0 + 8 * s);
                        mma_commit(tfull0 + 8 * b);
                        issued = true;
                    }
                }
                if (issued) {
                    // Every MMA must have finished before TMEM is released.
                    mma_commit(drain_bar);
                    if (!mbar_wait(drain_bar, 0, nullptr, budget)) atomicCAS(p.err, 0, DEV_TIMEOUT_DRAIN);
                }
            }
            __syncwarp();
        }
    } else {
        regs_inc<REGS_EPILOGUE>();
        // ---------------------------------------------------------------- epilogue
        const int quad = warp & 3;              // TMEM lanes 32*quad .. 32*quad + 31
        const int half = (warp - EPI_WARP0) >> 2;   // columns 128*half .. 128*half + 127
        const int r = quad * 32 + lane;         // row within the tile
        const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t j = 0;
        float acc[128];

        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            const TileInfo ti = decode_tile<GROUPED>(t, p, s_tstart, s_off);
            const int64_t row = ti.row0 + r;
            const bool row_ok = row >= 0 && row < ti.row_end;
            const int ncol0 = ti.n0 + half * 128;
            const bool blk_ok = ncol0 < p.N;
            const float* sa_ptr = p.a_s + (row_ok ? row : 0);
            const float* sw_ptr =
                p.w_s + (static_cast<int64_t>(ti.g) * p.NB + (blk_ok ? ncol0 / 128 : 0)) * KB;
            float sa_next = row_ok ? __ldg(sa_ptr) : 0.0f;
            float sw_next = blk_ok ? __ldg(sw_ptr) : 0.0f;

#pragma unroll
            for (int i = 0; i < 128; i++) acc[i] = 0.0f;

            bool ok = true;
            for (int kb = 0; kb < KB; kb++, j++) {
                const float sc = __fmul_rn(sa_next, sw_next);
                if (kb + 1 < KB) {
                    sa_next = row_ok ? __ldg(sa_ptr + static_cast<int64_t>(kb + 1) * p.rows) : 0.0f;
                    sw_next = blk_ok ? __ldg(sw_ptr + kb + 1) : 0.0f;
                }
                const uint32_t b = j & 1u;
                const uint32_t pb = (j >> 1) & 1u;
                const bool got = mbar_wait(tfull0 + 8 * b, pb, abort_flag, budget);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0) raise_error(p.err, abort_flag, DEV_TIMEOUT_EPILOGUE);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + t_lane + b * BN + half * 128;
#pragma unroll
                for (int c = 0; c < 4; c += 2) {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32cols(taddr + c * 32, v0);
                    tmem_ld_32cols(taddr + (c + 1) * 32, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        acc[c * 32 + i] = fmaf(__uint_as_float(v0[i]), sc, acc[c * 32 + i]);
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        acc[(c + 1) * 32 + i] =
                            fmaf(__uint_as_float(v1[i]), sc, acc[(c + 1) * 32 + i]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty0 + 8 * b);
            }
            if (!ok) break;

            if (row_ok) {
                if constexpr (OUT_F32) {
                    float* crow = static_cast<float*>(p.c) + row * p.ldc + ncol0;
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        if (ncol0 + 4 * i < p.N)
                            st_v4(crow + 4 * i, __float_as_uint(acc[4 * i]),
                                  __float_as_uint(acc[4 * i + 1]), __float_as_uint(acc[4 * i + 2]),
                                  __float_as_uint(acc[4 * i + 3]));
                } else {
                    uint16_t* crow = static_cast<uint16_t*>(p.c) + row * p.ldc + ncol0;
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        if (ncol0 + 8 * i < p.N)
                            st_v4(crow + 8 * i, pack_bf16x2(acc[8 * i], acc[8 * i + 1]),
                                  pack_bf16x2(acc[8 * i + 2], acc[8 * i + 3]),
                                  pack_bf16x2(acc[8 * i + 4], acc[8 * i + 5]),
                                  pack_bf16x2(acc[8 * i + 6], acc[8 * i + 7]));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) {
        __syncwarp();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <bool GROUPED, bool OUT_F32>
cudaError_t launch_one(const CUtensorMap& ma, const CUtensorMap& mb, const GemmArgs& args,
                       int grid, cudaStream_t stream)
{
    auto kern = fp8_blockscaled_gemm_kernel<GROUPED, OUT_F32>;
    const size_t smem = gemm_smem_bytes(GROUPED, args.G);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, THREADS, smem, stream>>>(ma, mb, args);
    return cudaGetLastError();
}

}  // namespace

size_t gemm_smem_bytes(bool grouped, int G)
{
    size_t bytes = static_cast<size_t>(GROUP_OFF) + ALIGN_PAD;
    if (grouped) bytes += 2 * static_cast<size_t>(G + 1) * sizeof(int);
    return bytes;
}

cudaError_t launch_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b, const GemmArgs& args,
                        bool grouped, bool out_f32, int grid, cudaStream_t stream)
{
    if (grouped)
        return out_f32 ? launch_one<true, true>(map_a, map_b, args, grid, stream)
                       : launch_one<true, false>(map_a, map_b, args, grid, stream);
    return out_f32 ? launch_one<false, true>(map_a, map_b, args, grid, stream)
                   : launch_one<false, false>(map_a, map_b, args, grid, stream);
}

}  // namespace fp8bs
