// gemm_small.cu -- the block-scaled FP8 GEMM C = A W^T of fp8_blockscaled_gemm for few rows of A
// (decode-size M <= 64), computed as C^T = W A^T ("swap AB"): the weight rows fill the tensor
// core's 128-row side and the M tokens its narrow N side (32 or 64 columns). When the
// weight tiles alone cannot cover the SMs, the K loop of a tile is split over a cluster of up to
// 8 CTAs, which add their FP32 partial tiles through distributed shared memory (no workspace).
//
// Arithmetic per output element as in gemm.cu (codingmall.com "Tăng độ chính xác tích lũy",
// dtcms.com 三.3): per 128-wide K block the tensor cores form P = sum_k dec(w[n][k]) dec(a[m][k])
// in FP32 and the epilogue adds fl(s_w[n/128][kb] * s_a[kb][m]) * P with one FMA, in increasing
// kb within a CTA's K range; a split cluster then adds its CTAs' partial sums in rank order.
//
// Roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer (and TMEM), warp 2 scale loader
// (the K block's column scales fl(s_w * s_a[m]) into a shared ring), warps 4-11 epilogue (TMEM lane
// quarter w % 4, column half (w - 4) / 4). Every wait is bounded as in gemm.cu; after the K loop
// all CTAs of a cluster always meet at two cluster barriers, whether or not a role gave up.
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

template <int BNT>   // tokens per tile
struct SmallLayout {
    static constexpr int A_BYTES = SM_BM * SM_BK;        // weight tile (the MMA's A operand)
    static constexpr int B_BYTES = BNT * SM_BK;          // token tile (the MMA's B operand)
    static constexpr int STAGE = A_BYTES + B_BYTES;
    // as many stages as fit in ~192 KB: the weight stream needs the bytes in flight
#ifdef FP8BS_SERIAL_PIPELINE
    // debug build (build.py --serial): the fewest stages whose ring still holds the partial tile
    static constexpr int STAGES = (SM_BM * BNT * 4 + STAGE - 1) / STAGE;
#else
    static constexpr int STAGES = (192 * 1024) / STAGE > 10 ? 10 : (192 * 1024) / STAGE;
#endif
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_BYTES;
    static constexpr int RING = STAGES * STAGE;
    static constexpr int PART_BYTES = SM_BM * BNT * 4;   // FP32 partial tile, [column][row]
    static_assert(PART_BYTES <= RING, "the partial tile reuses the operand ring");
    static_assert(B_BYTES % 1024 == 0, "token tiles keep 1024-byte alignment");
    static constexpr int SCL_OFF = RING;
    static constexpr int SLOT = BNT * 4 + 16;            // one K block's column scales + s_w
    static constexpr int BAR_OFF = SCL_OFF + SM_SLOTS * SLOT;
    // TMEM accumulators of BNT columns: as many as fit in half (32 tokens) or all (64, 128) of
    // the 512 columns, so that the MMAs run up to NBUF K blocks ahead of the epilogue and the
    // hand-over of a block's partial is hidden behind the weight stream (one in the serial build)
#ifdef FP8BS_SERIAL_PIPELINE
    static constexpr int NBUF = 1;
#else
    static constexpr int NBUF = BNT <= 64 ? 8 : 4;
#endif
    static constexpr uint32_t TMEM_COLS = NBUF * BNT;    // 256 or 512 (serial: BNT)
    // full[S], empty[S], tfull[NBUF], tempty[NBUF], drain, sfull[SLOTS], sempty[SLOTS]
    static constexpr int NUM_BARS = 2 * STAGES + 2 * NBUF + 1 + 2 * SM_SLOTS;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int BYTES = MISC_OFF + 16 + SM_ALIGN;
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

// A float in the shared memory of any CTA of the cluster (address from mapa_shared).
__device__ __forceinline__ float ld_cluster_f32(uint32_t cluster_addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}

template <int BNT, bool OUT_F32>
__global__ void __launch_bounds__(SM_THREADS, 1)
gemm_small_kernel(const __grid_constant__ CUtensorMap map_w,
                  const __grid_constant__ CUtensorMap map_a, const SmallArgs p)
{
    using L = SmallLayout<BNT>;
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
    const int S = p.split;
    const int rank = static_cast<int>(blockIdx.x) % S;   // == rank in the cluster of S CTAs
    const int item = static_cast<int>(blockIdx.x) / S;
    const int nt = item % p.n_tiles;
    const int mt = item / p.n_tiles;
    const int n0 = nt * SM_BM;
    const int m0 = mt * BNT;
    const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * p.KB / S);
    const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * p.KB / S);

    if (threadIdx.x == 0) {
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
    if (warp == SM_PRODUCER && lane == 0) {
        tma_prefetch_map(&map_w);
        tma_prefetch_map(&map_a);
    }
    if (warp == SM_MMA) {
        tmem_alloc(smem_u32(tmem_holder), L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == SM_PRODUCER) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; kb++, it++) {
                const uint32_t s = it % L::STAGES;
                if (!mbar_wait(empty0 + 8 * s, ((it / L::STAGES) & 1u) ^ 1u, abort_addr, budget)) {
                    raise_small(p.err, abort_addr, DEV_TIMEOUT_PRODUCER);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full0 + 8 * s, L::STAGE);
                tma_load_2d(sW + s * L::A_BYTES, &map_w, full0 + 8 * s, kb * SM_BK, n0);
                tma_load_2d(sA + s * L::B_BYTES, &map_a, full0 + 8 * s, kb * SM_BK, m0);
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
            bool issued = false;
            for (int kb = kb0; kb < kb1; kb++, it++) {
                const uint32_t b = it % L::NBUF;
                if (!mbar_wait(tempty0 + 8 * b, ((it / L::NBUF) & 1u) ^ 1u, abort_addr, budget)) {
                    raise_small(p.err, abort_addr, DEV_TIMEOUT_MMA_TMEM);
                    break;
                }
                const uint32_t s = it % L::STAGES;
                if (!mbar_wait(full0 + 8 * s, (it / L::STAGES) & 1u, abort_addr, budget)) {
                    raise_small(p.err, abort_addr, DEV_TIMEOUT_MMA_FULL);
                    break;
                }
                tc_fence_after();
                const uint64_t da = desc_kmajor_sw128(sW + s * L::A_BYTES);
                const uint64_t db = desc_kmajor_sw128(sA + s * L::B_BYTES);
                const uint32_t d_tmem = tmem_base + b * BNT;
#pragma unroll
                for (int k = 0; k < SM_BK / 32; k++)   // +32 bytes of K = +2 in the address field
                    mma_e4m3(d_tmem, da + 2 * k, db + 2 * k, IDESC, k > 0 ? 1u : 0u);
                mma_commit(empty0 + 8 * s);
                mma_commit(tfull0 + 8 * b);
                issued = true;
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
        for (int kb = kb0; kb < kb1; kb++, it++) {
            const uint32_t slot = it % SM_SLOTS;
            const bool got =
                mbar_wait(sempty0 + 8 * slot, ((it / SM_SLOTS) & 1u) ^ 1u, abort_addr, budget);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) raise_small(p.err, abort_addr, DEV_TIMEOUT_SCALES);
                break;
            }
            const uint32_t sl = scl0 + slot * L::SLOT;
            const float* a_row = p.a_s + static_cast<int64_t>(kb) * p.M + m0;
            for (int c = lane; c < BNT; c += 32) {
                const bool v = m0 + c < p.M;
                cp_async_4(sl + c * 4, v ? a_row + c : zero_src, v ? 4u : 0u);
            }
            if (lane == 0) cp_async_4(sl + BNT * 4, p.w_s + static_cast<int64_t>(nt) * p.KB + kb, 4u);
            cp_async_commit();
            if (it >= SCALE_AHEAD) {
                cp_async_wait_group<SCALE_AHEAD>();
                finish(fin++);
            }
        }
        cp_async_wait_group<0>();
        while (fin < it) finish(fin++);
    } else if (warp >= SM_EPI0) {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;                        // TMEM lanes 32 quad .. 32 quad + 31
        const int half = (warp - SM_EPI0) >> 2;           // columns HALF half .. + HALF - 1
        const int row = quad * 32 + lane;                 // weight row within the tile
        const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
        float acc[HALF];
#pragma unroll
        for (int c = 0; c < HALF; c++) acc[c] = 0.0f;
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1; kb++, it++) {
            const uint32_t slot = it % SM_SLOTS;
            const bool sgot = mbar_wait(sfull0 + 8 * slot, (it / SM_SLOTS) & 1u, abort_addr, budget);
            const uint32_t b = it % L::NBUF;
            const bool got =
                sgot && mbar_wait(tfull0 + 8 * b, (it / L::NBUF) & 1u, abort_addr, budget);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) raise_small(p.err, abort_addr, DEV_TIMEOUT_EPILOGUE);
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
                    acc[c0 + 4 * q] = __fmaf_rn(f32x2_lo(uu[2 * q]), s4[q].x, acc[c0 + 4 * q]);
                    acc[c0 + 4 * q + 1] = __fmaf_rn(f32x2_hi(uu[2 * q]), s4[q].y, acc[c0 + 4 * q + 1]);
                    acc[c0 + 4 * q + 2] = __fmaf_rn(f32x2_lo(uu[2 * q + 1]), s4[q].z, acc[c0 + 4 * q + 2]);
                    acc[c0 + 4 * q + 3] = __fmaf_rn(f32x2_hi(uu[2 * q + 1]), s4[q].w, acc[c0 + 4 * q + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(tempty0 + 8 * b);
                mbar_arrive(sempty0 + 8 * slot);
            }
        }
        // The last tfull wait covered every MMA, so the operand ring is no longer read: the
        // partial tile goes there, column-major (a warp writes 32 consecutive floats per column).
#pragma unroll
        for (int c = 0; c < HALF; c++)
            st_shared_f32s(base + ((half * HALF + c) * SM_BM + row) * 4, acc[c]);
    }

    // ---------------------------------------------------------------- split-K reduction
    // Every thread of every CTA of the cluster runs this, whatever happened above.
    tc_fence_before();
    __syncthreads();
    if (S > 1) cluster_sync();              // the peers' partial tiles are written and visible
    const int rows = SM_BM / S;
    const int r_lo = rank * rows;
    for (int idx = threadIdx.x; idx < rows * BNT; idx += SM_THREADS) {
        const int r = r_lo + idx % rows;    // consecutive threads: consecutive output columns n
        const int c = idx / rows;
        const uint32_t off = base + (c * SM_BM + r) * 4;
        float v = 0.0f;
        if (S > 1) {
            for (int j = 0; j < S; j++) v += ld_cluster_f32(mapa_shared(off, static_cast<uint32_t>(j)));
        } else {
            v += *reinterpret_cast<const float*>(smem + (c * SM_BM + r) * 4);
        }
        const int64_t m = m0 + c;
        const int64_t n = n0 + r;
        if (m < p.M && n < p.N) {
            if constexpr (OUT_F32) {
                static_cast<float*>(p.c)[m * p.ldc + n] = v;
            } else {
                static_cast<uint16_t*>(p.c)[m * p.ldc + n] = bf16_rn(v);
            }
        }
    }
    if (S > 1) cluster_sync();              // no CTA leaves while a peer still reads its tile
    tc_fence_after();
    if (warp == SM_MMA) {
        __syncwarp();
        tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

template <int BNT, bool OUT_F32>
cudaError_t launch_small(const CUtensorMap& mw, const CUtensorMap& ma, const SmallArgs& args,
                         cudaStream_t stream)
{
    auto kern = gemm_small_kernel<BNT, OUT_F32>;
    const size_t smem = SmallLayout<BNT>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(args.split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(args.n_tiles * args.m_tiles * args.split));
    cfg.blockDim = dim3(SM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mw, ma, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

int gemm_small_tokens(int64_t M) { return M <= 32 ? 32 : 64; }

cudaError_t launch_gemm_small(const CUtensorMap& map_w, const CUtensorMap& map_a,
                              const SmallArgs& args, int bnt, bool out_f32, cudaStream_t stream)
{
    if (bnt == 32)
        return out_f32 ? launch_small<32, true>(map_w, map_a, args, stream)
                       : launch_small<32, false>(map_w, map_a, args, stream);
    return out_f32 ? launch_small<64, true>(map_w, map_a, args, stream)
                   : launch_small<64, false>(map_w, map_a, args, stream);
}

}  // namespace fp8bs
