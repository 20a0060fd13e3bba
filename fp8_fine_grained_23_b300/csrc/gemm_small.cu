// gemm_small.cu -- the block-scaled FP8 GEMM C = A W^T of fp8_blockscaled_gemm for few rows of A
// (decode-size M <= 64), computed as C^T = W A^T ("swap AB"): the weight rows fill the tensor
// core's 128-row side and the M tokens its narrow N side (32 or 64 columns). When the
// weight tiles alone cannot cover the SMs, the K loop of a tile is split over a cluster of up to
// 8 CTAs: each CTA deposits the rows of its FP32 partial tile in the shared memory of the CTA
// that sums them (distributed shared memory, no workspace). Otherwise the grid is persistent
// (at most one CTA per SM, items taken in turn) and each tile's sums go from registers to C.
//
// Arithmetic per output element as in gemm.cu (codingmall.com "Tăng độ chính xác tích lũy",
// dtcms.com 三.3): per 128-wide K block the tensor cores form P = sum_k dec(w[n][k]) dec(a[m][k])
// in FP32 and the epilogue adds fl(s_w[n/128][kb] * s_a[kb][m]) * P with one FMA, in increasing
// kb within a CTA's K range; a split cluster then adds its CTAs' partial sums in rank order.
//
// Roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer (and TMEM), warp 2 scale loader
// (the K block's column scales fl(s_w * s_a[m]) into a shared ring), warps 4-11 epilogue (TMEM lane
// quarter w % 4, column half (w - 4) / 4). Every wait is bounded as in gemm.cu; a split cluster's
// CTAs always meet at its cluster barriers, whether or not a role gave up.
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {

namespace {

constexpr int SM_BM = 128;        // weight rows per tile (the MMA's M)
constexpr int SM_BK = 128;
constexpr int SM_SLOTS = 8;
constexpr int SM_THREADS = 384;
constexpr int SM_PRODUCER = 0;
constexpr int SM_MMA = 1;
constexpr int SM_SCALE = 2;
constexpr int SM_EPI0 = 4;
constexpr int SM_EPI_WARPS = 8;
constexpr int SM_ALIGN = 1024;

constexpr int SM_SMEM_MAX = 227 * 1024;   // dynamic shared memory a CTA may opt in to
constexpr int SM_MAX_STAGES = 10;

template <int BNT, bool SPLIT>   // tokens per tile; split-K over a cluster
struct SmallLayout {
    static constexpr int A_BYTES = SM_BM * SM_BK;        // weight tile (the MMA's A operand)
    static constexpr int B_BYTES = BNT * SM_BK;          // token tile (the MMA's B operand)
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static_assert(B_BYTES % 1024 == 0, "token tiles keep 1024-byte alignment");
    // Split-K: the region in which the S CTAs of a cluster deposit the rows of their partial
    // tiles that this CTA sums: [source rank][token column][128 / S rows], 128 x BNT FP32.
    static constexpr int PART_BYTES = SPLIT ? SM_BM * BNT * 4 : 0;
    static constexpr int SLOT = BNT * 4 + 16;            // one K block's column scales + s_w
    // TMEM accumulators of BNT columns: as many as fit in half (32 tokens) or all (64, 128) of
    // the 512 columns, so that the MMAs run up to NBUF K blocks ahead of the epilogue and the
    // hand-over of a block's partial is hidden behind the weight stream (one in the serial build)
#ifdef FP8BS_SERIAL_PIPELINE
    static constexpr int NBUF = 1;
#else
    static constexpr int NBUF = BNT <= 64 ? 8 : 4;
#endif
    static constexpr uint32_t TMEM_COLS = NBUF * BNT;    // 256 or 512 (serial: BNT)
#ifdef FP8BS_SERIAL_PIPELINE
    static constexpr int STAGES = 1;   // debug build (build.py --serial): one stage
#else
    // everything but the operand ring, with barriers for the most stages
    static constexpr int FIXED = PART_BYTES + SM_SLOTS * SLOT +
                                 (2 * SM_MAX_STAGES + 2 * NBUF + 1 + 2 * SM_SLOTS) * 8 + 16 +
                                 SM_ALIGN;
    // as many stages as fit in ~192 KB (the weight stream needs the bytes in flight), or, beside
    // the split-K region, in what is left of the CTA's shared memory
    static constexpr int FIT = (SPLIT ? SM_SMEM_MAX - FIXED : 192 * 1024) / STAGE;
    static constexpr int STAGES = FIT > SM_MAX_STAGES ? SM_MAX_STAGES : FIT;
#endif
    static_assert(STAGES >= 1 && STAGES <= SM_MAX_STAGES, "operand ring");
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_BYTES;
    static constexpr int RING = STAGES * STAGE;
    static constexpr int PART_OFF = RING;
    static constexpr int SCL_OFF = PART_OFF + PART_BYTES;
    static constexpr int BAR_OFF = SCL_OFF + SM_SLOTS * SLOT;
    // full[S], empty[S], tfull[NBUF], tempty[NBUF], drain, sfull[SLOTS], sempty[SLOTS]
    static constexpr int NUM_BARS = 2 * STAGES + 2 * NBUF + 1 + 2 * SM_SLOTS;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int BYTES = MISC_OFF + 16 + SM_ALIGN;
    static_assert(BYTES <= SM_SMEM_MAX, "shared memory");
    static_assert(SLOT % 16 == 0 && PART_BYTES % 16 == 0, "16-byte aligned regions");
};

__device__ __forceinline__ void raise_small(int* err, uint32_t abort_addr, int code)
{
    st_shared_volatile_u32(abort_addr, 1u);
    atomicCAS(err, 0, code);
}

__device__ __forceinline__ void st_shared_f32s(uint32_t addr, float v)
{
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ float ld_shared_f32s(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's most recent cp.async groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float4 ld_shared_f32x4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint16_t bf16_rn(float v)
{
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
    return r;
}

// Split-phase cluster barrier (every thread of every CTA of the cluster): arrive without ordering
// any memory operation, and the matching wait.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// A float into the shared memory of any CTA of the cluster (address from mapa_shared).
__device__ __forceinline__ void st_cluster_f32(uint32_t cluster_addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}

// Four consecutive outputs of one row of C (16-byte aligned for FP32, 8-byte for BF16).
template <bool OUT_F32>
__device__ __forceinline__ void st_out4(void* dst, float4 v)
{
    if constexpr (OUT_F32) {
        asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(v.x), "f"(v.y),
                     "f"(v.z), "f"(v.w)
                     : "memory");
    } else {
        const uint32_t lo = static_cast<uint32_t>(bf16_rn(v.x)) | (static_cast<uint32_t>(bf16_rn(v.y)) << 16);
        const uint32_t hi = static_cast<uint32_t>(bf16_rn(v.z)) | (static_cast<uint32_t>(bf16_rn(v.w)) << 16);
        asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(dst), "r"(lo), "r"(hi) : "memory");
    }
}

// SPLIT: a cluster per item, K split over its CTAs; PERSIST: more items than CTAs, taken in turn;
// neither: one item per CTA.
template <int BNT, bool OUT_F32, bool SPLIT, bool PERSIST>
__global__ void __launch_bounds__(SM_THREADS, 1)
gemm_small_kernel(const __grid_constant__ CUtensorMap map_w,
                  const __grid_constant__ CUtensorMap map_a, const SmallArgs p)
{
    using L = SmallLayout<BNT, SPLIT>;
    constexpr int HALF = BNT / 2;                        // columns per epilogue thread
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + (SM_ALIGN - 1)) & ~static_cast<uint32_t>(SM_ALIGN - 1);
    uint8_t* smem = smem_raw + (base - raw);

    const uint32_t sW = base + L::A_OFF;
    const uint32_t sA = base + L::B_OFF;
    const uint32_t full0 = base + L::BAR_OFF;
    const uint32_t empty0 = full0 + 8 * L::STAGES;
    const uint32_t tfull0 = empty0 + 8 * L::STAGES;
    const uint32_t tempty0 = tfull0 + 8 * L::NBUF;
    const uint32_t drain_bar = tempty0 + 8 * L::NBUF;
    const uint32_t sfull0 = drain_bar + 8;
    const uint32_t sempty0 = sfull0 + 8 * SM_SLOTS;
    const uint32_t scl0 = base + L::SCL_OFF;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
    const uint32_t abort_addr = base + L::MISC_OFF + 4;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long budget = p.budget;
    const int S = SPLIT ? p.split : 1;
    const int rank = static_cast<int>(blockIdx.x) % S;   // == rank in the cluster of S CTAs
    // Work items (weight tile nt, token tile mt), t = mt * n_tiles + nt. A split cluster takes
    // one item and CTA `rank` its share of the K loop. A persistent CTA b takes items b,
    // b + gridDim.x, ... with the whole K loop each, its pipelines running on from one item into
    // the next; the item loops below end after one pass otherwise.
    static_assert(!(SPLIT && PERSIST), "a split cluster takes one item");
    const int items = p.n_tiles * p.m_tiles;
    const int t_first = static_cast<int>(blockIdx.x) / S;
    const int t_step = static_cast<int>(gridDim.x);
    const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * p.KB / S);
    const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * p.KB / S);

    if (threadIdx.x == 0) {
        tma_prefetch_map(&map_w);
        tma_prefetch_map(&map_a);
        for (int s = 0; s < L::STAGES; s++) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < L::NBUF; b++) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, SM_EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        for (int i = 0; i < SM_SLOTS; i++) {
            mbar_init(sfull0 + 8 * i, 32);               // every loader lane, after its stores
            mbar_init(sempty0 + 8 * i, SM_EPI_WARPS);
        }
        st_shared_volatile_u32(abort_addr, 0u);
        fence_mbar_init();
    }
    if (warp == SM_MMA) {
        tmem_alloc(smem_u32(tmem_holder), L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // Split-K: a CTA writes into its peers' shared memory only once every CTA of the cluster is
    // known to be running; that phase of the cluster barrier completes long before the first
    // such write (the epilogue waits for it just before, every other warp after its role).
    if constexpr (SPLIT) cluster_arrive_relaxed();

    if (warp == SM_PRODUCER) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = t_first; ok && t < items; t += t_step) {
                const int n0 = (t % p.n_tiles) * SM_BM;
                const int m0 = (t / p.n_tiles) * BNT;
                for (int kb = kb0; kb < kb1; kb++, it++) {
                    const uint32_t s = it % L::STAGES;
                    if (!mbar_wait(empty0 + 8 * s, ((it / L::STAGES) & 1u) ^ 1u, abort_addr,
                                   budget)) {
                        raise_small(p.err, abort_addr, DEV_TIMEOUT_PRODUCER);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full0 + 8 * s, L::STAGE);
                    tma_load_2d(sW + s * L::A_BYTES, &map_w, full0 + 8 * s, kb * SM_BK, n0);
                    tma_load_2d(sA + s * L::B_BYTES, &map_a, full0 + 8 * s, kb * SM_BK, m0);
                }
                if constexpr (!PERSIST) break;
            }
            if (!ok || ld_shared_volatile_u32(abort_addr) != 0) {
                // the MMA side may never consume what is in flight: wait for the last copy
                // issued into every stage before the CTA may exit
                const uint32_t first = it > L::STAGES ? it - L::STAGES : 0;
                for (uint32_t i = first; i < it; i++)
                    if (!mbar_wait(full0 + 8 * (i % L::STAGES), (i / L::STAGES) & 1u, 0u, budget))
                        atomicCAS(p.err, 0, DEV_TIMEOUT_DRAIN);
            }
        }
    } else if (warp == SM_MMA) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_e4m3_f32(SM_BM, BNT);
            uint32_t it = 0;
            bool issued = false, ok = true;
            for (int t = t_first; ok && t < items; t += t_step) {
                for (int kb = kb0; kb < kb1; kb++, it++) {
                    const uint32_t b = it % L::NBUF;
                    if (!mbar_wait(tempty0 + 8 * b, ((it / L::NBUF) & 1u) ^ 1u, abort_addr,
                                   budget)) {
                        raise_small(p.err, abort_addr, DEV_TIMEOUT_MMA_TMEM);
                        ok = false;
                        break;
                    }
                    const uint32_t s = it % L::STAGES;
                    if (!mbar_wait(full0 + 8 * s, (it / L::STAGES) & 1u, abort_addr, budget)) {
                        raise_small(p.err, abort_addr, DEV_TIMEOUT_MMA_FULL);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = desc_kmajor_sw128(sW + s * L::A_BYTES);
                    const uint64_t db = desc_kmajor_sw128(sA + s * L::B_BYTES);
                    const uint32_t d_tmem = tmem_base + b * BNT;
#pragma unroll
                    for (int k = 0; k < SM_BK / 32; k++)   // +32 bytes of K = +2 in the address
                        mma_e4m3(d_tmem, da + 2 * k, db + 2 * k, IDESC, k > 0 ? 1u : 0u);
                    mma_commit(empty0 + 8 * s);
                    mma_commit(tfull0 + 8 * b);
                    issued = true;
                }
                if constexpr (!PERSIST) break;
            }
            if (issued) {
                mma_commit(drain_bar);   // every MMA has finished before TMEM is released
                if (!mbar_wait(drain_bar, 0, 0u, budget)) atomicCAS(p.err, 0, DEV_TIMEOUT_DRAIN);
            }
        }
    } else if (warp == SM_SCALE) {
        // ------------------------------------------------------------ column scales
        // The K block's token scales s_a[kb][m0 ..] (zero past M) and its weight-block scale
        // stream into a slot by cp.async, SCALE_AHEAD blocks ahead of the block being finished;
        // once a block's copies have landed the slot's BNT products fl(s_w * s_a[m]) are formed
        // in place and the slot is handed to the epilogue. (Plain loads here exposed two
        // dependent L2/HBM latencies per K block, which paced the whole kernel.)
        constexpr int SCALE_AHEAD = SM_SLOTS - 2;
        const float* zero_src = p.a_s;   // any valid address: zero-filled copies read nothing
        uint32_t it = 0, fin = 0;
        auto finish = [&](uint32_t jt) {
            const uint32_t sl = scl0 + (jt % SM_SLOTS) * L::SLOT;
            __syncwarp();                                  // lane 0's copy of s_w is visible
            const float sw = ld_shared_f32s(sl + BNT * 4);
            for (int c = lane; c < BNT; c += 32)
                st_shared_f32s(sl + c * 4, __fmul_rn(sw, ld_shared_f32s(sl + c * 4)));
            mbar_arrive(sfull0 + 8 * (jt % SM_SLOTS));
        };
        bool ok = true;
        for (int t = t_first; ok && t < items; t += t_step) {
            const int nt = t % p.n_tiles;
            const int m0 = (t / p.n_tiles) * BNT;
            for (int kb = kb0; kb < kb1; kb++, it++) {
                const uint32_t slot = it % SM_SLOTS;
                const bool got = mbar_wait(sempty0 + 8 * slot, ((it / SM_SLOTS) & 1u) ^ 1u,
                                           abort_addr, budget);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0) raise_small(p.err, abort_addr, DEV_TIMEOUT_SCALES);
                    ok = false;
                    break;
                }
                const uint32_t sl = scl0 + slot * L::SLOT;
                const float* a_row = p.a_s + static_cast<int64_t>(kb) * p.M + m0;
                for (int c = lane; c < BNT; c += 32) {
                    const bool v = m0 + c < p.M;
                    cp_async_4(sl + c * 4, v ? a_row + c : zero_src, v ? 4u : 0u);
                }
                if (lane == 0)
                    cp_async_4(sl + BNT * 4, p.w_s + static_cast<int64_t>(nt) * p.KB + kb, 4u);
                cp_async_commit();
                if (it >= SCALE_AHEAD) {
                    cp_async_wait_group<SCALE_AHEAD>();
                    finish(fin++);
                }
            }
            if constexpr (!PERSIST) break;
        }
        cp_async_wait_group<0>();
        while (fin < it) finish(fin++);
    } else if (warp >= SM_EPI0) {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;                        // TMEM lanes 32 quad .. 32 quad + 31
        const int half = (warp - SM_EPI0) >> 2;           // columns HALF half .. + HALF - 1
        const int row = quad * 32 + lane;                 // weight row within the tile
        const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t it = 0;
        bool ok = true;
        // (a split cluster's CTA runs this loop once, so its epilogue waits on the cluster
        // barrier exactly once, as every other warp does below; t_first < items always)
        for (int t = t_first; ok && t < items; t += t_step) {
            const int n0 = (t % p.n_tiles) * SM_BM;
            const int m0 = (t / p.n_tiles) * BNT;
            float acc[HALF];
#pragma unroll
            for (int c = 0; c < HALF; c++) acc[c] = 0.0f;
            for (int kb = kb0; kb < kb1; kb++, it++) {
                const uint32_t slot = it % SM_SLOTS;
                const bool sgot =
                    mbar_wait(sfull0 + 8 * slot, (it / SM_SLOTS) & 1u, abort_addr, budget);
                const uint32_t b = it % L::NBUF;
                const bool got =
                    sgot && mbar_wait(tfull0 + 8 * b, (it / L::NBUF) & 1u, abort_addr, budget);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0) raise_small(p.err, abort_addr, DEV_TIMEOUT_EPILOGUE);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + t_lane + b * BNT + half * HALF;
                const uint32_t sc = scl0 + slot * L::SLOT + half * HALF * 4;
                // 16-column chunks, the next chunk's TMEM load and this chunk's scale loads in
                // flight while the previous chunk is promoted
                uint64_t u[2][8];
                tmem_ld_16cols(taddr, u[0]);
#pragma unroll
                for (int ch = 0; ch < HALF / 16; ch++) {
                    const int c0 = 16 * ch;
                    float4 s4[4];
#pragma unroll
                    for (int q = 0; q < 4; q++) s4[q] = ld_shared_f32x4(sc + (c0 + 4 * q) * 4);
                    tmem_wait_ld(u[ch & 1]);
                    if (ch + 1 < HALF / 16) tmem_ld_16cols(taddr + c0 + 16, u[(ch + 1) & 1]);
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const uint64_t* uu = u[ch & 1];
                        float* a4 = acc + c0 + 4 * q;
                        a4[0] = __fmaf_rn(f32x2_lo(uu[2 * q]), s4[q].x, a4[0]);
                        a4[1] = __fmaf_rn(f32x2_hi(uu[2 * q]), s4[q].y, a4[1]);
                        a4[2] = __fmaf_rn(f32x2_lo(uu[2 * q + 1]), s4[q].z, a4[2]);
                        a4[3] = __fmaf_rn(f32x2_hi(uu[2 * q + 1]), s4[q].w, a4[3]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(tempty0 + 8 * b);
                    mbar_arrive(sempty0 + 8 * slot);
                }
            }
            if constexpr (!SPLIT) {
                // The CTA owns the whole K loop: its sums are final and go straight from
                // registers to C (one store instruction of a warp covers 32 consecutive n of
                // one token row).
                const int64_t n = n0 + row;
#pragma unroll
                for (int c = 0; c < HALF; c++) {
                    const int64_t m = m0 + half * HALF + c;
                    if (m < p.M && n < p.N) {
                        if constexpr (OUT_F32) {
                            static_cast<float*>(p.c)[m * p.ldc + n] = acc[c];
                        } else {
                            static_cast<uint16_t*>(p.c)[m * p.ldc + n] = bf16_rn(acc[c]);
                        }
                    }
                }
            } else {
                // Weight row `row` is summed by the CTA of rank row / (128 / S): this CTA's
                // partial values of it go to that CTA's split-K region, in the slot of this
                // CTA's rank (a warp writes runs of consecutive rows of one column).
                cluster_wait();
                const int rows = SM_BM / S;
                const uint32_t dst = mapa_shared(
                    base + L::PART_OFF + ((rank * BNT + half * HALF) * rows + row % rows) * 4,
                    static_cast<uint32_t>(row / rows));
#pragma unroll
                for (int c = 0; c < HALF; c++) st_cluster_f32(dst + c * rows * 4, acc[c]);
            }
            if constexpr (!PERSIST) break;
        }
    }

    // ---------------------------------------------------------------- split-K reduction
    // Every thread of every CTA of the cluster runs this, whatever happened above.
    if constexpr (SPLIT) {
        if (warp < SM_EPI0) cluster_wait();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (SPLIT) {
        // Every CTA has deposited its rows and arrived (release) before any CTA passes (acquire),
        // and no CTA touches another's shared memory after this point, so one barrier suffices.
        cluster_sync();
        // CTA `rank` sums weight rows [rank * rows, + rows) over the S deposited partials, four
        // rows at a time, in rank order.
        const int n0 = (t_first % p.n_tiles) * SM_BM;
        const int m0 = (t_first / p.n_tiles) * BNT;
        const int rows = SM_BM / S;
        const int groups = rows / 4;        // per token column
        for (int idx = threadIdx.x; idx < groups * BNT; idx += SM_THREADS) {
            const int c = idx / groups;     // token column
            const int rl = 4 * (idx % groups);
            const int r = rank * rows + rl;
            float4 part[8];
#pragma unroll
            for (int j = 0; j < 8; j++)
                if (j < S)
                    part[j] = ld_shared_f32x4(base + L::PART_OFF + ((j * BNT + c) * rows + rl) * 4);
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if (j < S) {
                    v.x += part[j].x;
                    v.y += part[j].y;
                    v.z += part[j].z;
                    v.w += part[j].w;
                }
            }
            const int64_t m = m0 + c;
            const int64_t n = n0 + r;       // n % 4 == 0 and N % 16 == 0: all four or none
            if (m < p.M && n < p.N) {
                if constexpr (OUT_F32) {
                    st_out4<true>(static_cast<float*>(p.c) + m * p.ldc + n, v);
                } else {
                    st_out4<false>(static_cast<uint16_t*>(p.c) + m * p.ldc + n, v);
                }
            }
        }
    }
    tc_fence_after();
    if (warp == SM_MMA) {
        __syncwarp();
        tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

template <int BNT, bool OUT_F32, bool SPLIT, bool PERSIST>
cudaError_t launch_small(const CUtensorMap& mw, const CUtensorMap& ma, const SmallArgs& args,
                         int max_ctas, cudaStream_t stream)
{
    auto kern = gemm_small_kernel<BNT, OUT_F32, SPLIT, PERSIST>;
    const size_t smem = SmallLayout<BNT, SPLIT>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(args.split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // split: one cluster of `split` CTAs per item; persistent: one CTA per SM; else one per item
    const int items = args.n_tiles * args.m_tiles;
    cfg.gridDim = dim3(static_cast<unsigned>(SPLIT ? items * args.split
                                                   : (PERSIST ? max_ctas : items)));
    cfg.blockDim = dim3(SM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mw, ma, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// split K over a cluster; more items than SMs: persistent; else one CTA per item
template <int BNT, bool OUT_F32>
cudaError_t launch_mode(const CUtensorMap& mw, const CUtensorMap& ma, const SmallArgs& args,
                        int max_ctas, cudaStream_t stream)
{
    if (args.split > 1) return launch_small<BNT, OUT_F32, true, false>(mw, ma, args, max_ctas, stream);
    if (args.n_tiles * args.m_tiles > max_ctas)
        return launch_small<BNT, OUT_F32, false, true>(mw, ma, args, max_ctas, stream);
    return launch_small<BNT, OUT_F32, false, false>(mw, ma, args, max_ctas, stream);
}

}  // namespace

int gemm_small_tokens(int64_t M) { return M <= 32 ? 32 : 64; }

cudaError_t launch_gemm_small(const CUtensorMap& map_w, const CUtensorMap& map_a,
                              const SmallArgs& args, int bnt, bool out_f32, int max_ctas,
                              cudaStream_t stream)
{
    if (bnt == 32)
        return out_f32 ? launch_mode<32, true>(map_w, map_a, args, max_ctas, stream)
                       : launch_mode<32, false>(map_w, map_a, args, max_ctas, stream);
    return out_f32 ? launch_mode<64, true>(map_w, map_a, args, max_ctas, stream)
                   : launch_mode<64, false>(map_w, map_a, args, max_ctas, stream);
}

}  // namespace fp8bs
