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
//   warp 0     TMA producer: streams the CTA's 128x128 A code tile and its part of the W code
//              tile into a shared-memory ring (128-byte swizzle), completion on mbarriers;
//   warp 1     TMEM owner and MMA issuer: per K block, four tcgen05.mma (K = 32 each,
//              kind::f8f6f4, E4M3 x E4M3 -> FP32) into one of two TMEM accumulators, then
//              tcgen05.commit to free the shared-memory stage and to hand the partial to the
//              epilogue;
//   warp 2     scale loader: per K block, cp.async copies of the tile's 128 activation scales
//              and its two weight-block scales into an 8-slot shared-memory ring (sfull/sempty
//              mbarriers), so the epilogue reads its scale from shared memory;
//   warp 3     store warp of the DEFER variant (dense BF16 or E4M3-code output, long K
//              loops): writes each output tile the epilogue staged in shared memory to C while
//              the epilogue works on the next tile; idle otherwise (warp 0 also builds the group
//              table of the grouped variant, whose tiles follow that table of device offsets);
//   warps 4-11 epilogue: warp w reads TMEM lanes 32*(w%4).. (its rows) and the 128 columns
//              128*((w-4)/4).. (one weight block). Per K block it loads the partial in 16- or
//              32-column pieces (the next piece in flight while the current one is promoted)
//              and promotes it into 128 FP32 registers per thread (packed pairs,
//              fma.rn.f32x2). At the end of the tile the results are staged in shared memory as
//              blocks of 32 rows x 64 bytes and leave as whole 64-byte row segments: through the
//              store warp, as TMA bulk stores, or as plain stores (BF16 or FP32).
//
// The dense GEMM runs on CTA pairs (clusters of two, cta_group::2): the pair computes a 256x256
// tile with one 256-row MMA per K step, issued by the even CTA. Each CTA loads only its own 128
// A rows and 128 of the 256 W rows, so a K block brings 32 KB into each SM instead of 48 KB; a
// stage takes 32 KB and four of them (as fast as six) leave room for a staged 64 KB output tile.
// Both CTAs' loads complete on the even CTA's
// `full` barrier; the MMA commits are multicast to both CTAs' `empty` and `tfull` barriers. The
// epilogue warps of both CTAs release a TMEM buffer on the even CTA's `tempty` barrier (the odd
// CTA's by remote arrives; in the row-scaled variant, whose epilogue has no register to spare,
// the odd CTA's otherwise idle MMA warp forwards its local release instead).
// The per-K-block hand-over of the partial through TMEM is what bounds this kernel: two buffers
// hold 1024 MMA cycles, less than the chain MMA completion -> drain -> release -> next MMA.
// The grouped GEMM, which is bound
// by streaming expert weights from HBM, keeps single-CTA MMAs on 128x256 tiles.
//
// Variants of the same kernel (template flags):
//   RS   (dense) B carries a scale per row and K block (the backward weight-gradient GEMM):
//        the scale ring holds the tile's 256 B-row scales and the promotion is
//        acc = fma(P * s_b[n], s_a[m], acc), in 16-column TMEM chunks;
//   SW   (grouped) gate and up weight rows interleaved per 128: a thread promotes 64 gate and the
//        matching 64 up columns, forms silu(gate) * up, exchanges row maxima with the partner
//        warp of its lane quarter and stores E4M3 codes with 1x128 scales;
//   QO   (dense) the output re-quantized to E4M3 in 1x128 tiles: a thread's 128 columns are one
//        tile, so amax, scale and codes are thread-local;
//   DEFER (dense, BF16 output or QO) output tiles written by the store warp (chosen by the host
//        for K loops of 32+ blocks and 4+ tiles per pair; otherwise TMA bulk stores for BF16, plain
//        stores for QO).
// (Few rows of A, M <= 64, go to the swap-AB kernel in gemm_small.cu instead.)
//
// Registers: the launch gives 168 per thread (65536 / 384, rounded to 8). Warpgroup 0 drops to
// 72 and the two epilogue warpgroups rise to 216 (128*72 + 256*216 = 384*168), which holds the
// 128 accumulators of an epilogue thread and its TMEM load registers (32 or 64).
// Every mbarrier wait is bounded (clock budget); on expiry the CTA records an error code in the
// device error word, stops issuing work, waits for its in-flight copies and MMAs, frees TMEM and
// returns.
#include <cstdint>

#include "e4m3.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {

namespace {

constexpr int BM = GEMM_BM;
constexpr int BN = GEMM_BN;
constexpr int BK = GEMM_BK;
constexpr int NUM_EPI_WARPS = 8;
constexpr int PRODUCER_WARP = 0;
constexpr int MMA_WARP = 1;
constexpr int SCALE_WARP = 2;
constexpr int STORE_WARP = 3;   // dense BF16 output: writes each staged output tile to C
constexpr int EPI_WARP0 = 4;
constexpr int THREADS = 384;
constexpr int REGS_CONTROL = 72;           // warpgroup 0 after setmaxnreg.dec
constexpr int REGS_EPILOGUE = 216;         // warpgroups 1 and 2 after setmaxnreg.inc
static_assert(128 * REGS_CONTROL + 256 * REGS_EPILOGUE == THREADS * 168,
              "register split must equal the launch allocation of 168 per thread");
// FP8BS_SERIAL_PIPELINE (a debug build, see build.py --serial): one operand stage, one scale
// slot and one TMEM accumulator, so that every role waits for the previous one at every K block;
// results must not change.
#ifdef FP8BS_SERIAL_PIPELINE
constexpr bool SERIAL = true;
#else
constexpr bool SERIAL = false;
#endif
constexpr int TMEM_BUFS = SERIAL ? 1 : 2;  // FP32 accumulators of 128 lanes x BN columns
constexpr int TMEM_COLS = TMEM_BUFS * BN;

constexpr int A_BYTES = BM * BK;           // E4M3: one byte per element
constexpr int B_BYTES = BN * BK;           // the whole W tile
constexpr int STG_WARP_BYTES = 32 * 64;    // output staging per epilogue warp: 32 rows x 64 B
constexpr int STG_BYTES = NUM_EPI_WARPS * STG_WARP_BYTES;
constexpr int SCALE_SLOTS = SERIAL ? 1 : 8;   // scale ring: one slot per K block in flight
constexpr int SCALE_SLOT_BYTES_BLOCK = 528;   // 128 activation scales + 2 weight-block scales
constexpr int SCALE_SLOT_BYTES_ROWS = 1536;   // 128 A-row scales + 256 B-row scales
constexpr int ALIGN_PAD = 1024;            // 128-byte-swizzled tiles need 1024-byte alignment

// Shared-memory layout per CTA. PAIR: a CTA holds its A tile and half of the W tile.
// RS: the B operand has a scale per row and K block (the 1d1d GEMM) instead of per 128x128 block.
// SW: the SwiGLU + re-quantizing epilogue, which exchanges row maxima between the two warps that
// share a 1x128 output tile (two tile-parity buffers x two halves x 128 rows of FP32).
template <bool GROUPED, bool PAIR, bool RS, bool SW = false>
struct Layout {
    static constexpr int SLOT = RS ? SCALE_SLOT_BYTES_ROWS : SCALE_SLOT_BYTES_BLOCK;
    static constexpr int CL = PAIR ? 2 : 1;              // CTAs per cluster
    static constexpr int B_PART = B_BYTES / CL;          // W rows held by this CTA
    static constexpr int STAGE = A_BYTES + B_PART;
    // (CTA pairs: 4 stages measured as fast as 6, which leaves room for a whole output tile)
    static constexpr int STAGES = SERIAL ? 1 : 4;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_BYTES;
    static constexpr int STG_OFF = STAGES * STAGE;
    // output staging: CTA pairs hold a whole BF16 output tile (4 boxes of 32 rows x 64 B per
    // epilogue warp), the grouped kernel one box per warp
    static constexpr int STG_SIZE = PAIR ? 4 * STG_BYTES : STG_BYTES;
    static constexpr int SCL_OFF = STG_OFF + STG_SIZE;
    static constexpr int XCH_OFF = SCL_OFF + SCALE_SLOTS * SLOT;
    static constexpr int BAR_OFF = XCH_OFF + (SW ? 2 * 2 * 128 * 4 : 0);
    // full[S], empty[S], tfull[2], tempty[2], drain, sfull[SCALE_SLOTS], sempty[SCALE_SLOTS],
    // ostaged, ofree (the output tile handed between the epilogue and the store warp),
    // SW: xch[4] (one per TMEM lane quarter)
    static constexpr int NUM_BARS = 2 * STAGES + 7 + 2 * SCALE_SLOTS + (SW ? 4 : 0);
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int GROUP_OFF = MISC_OFF + 16;
    static_assert(A_BYTES % 1024 == 0 && B_PART % 1024 == 0, "tiles keep 1024-byte alignment");
};

struct TileInfo {
    int64_t row0;      // first row of the tile in A / C
    int64_t row_end;   // rows >= row_end are not stored (next group or past the end)
    int64_t wrow0;     // first row of the W code tile (group * N + n0)
    int n0;            // first output column
    int g;             // group (0 for dense)
};

__device__ __forceinline__ void raise_error(int* err, uint32_t abort_addr, int code)
{
    st_shared_volatile_u32(abort_addr, 1u);
    atomicCAS(err, 0, code);
}

// Work item t of a CTA whose rank in its cluster is `crank`. Dense: t numbers groups of CL
// adjacent m-tiles (one per CTA of the cluster) on one n-tile. The m-groups are cut into bands of
// p.band; the items run band by band, and within a band m fastest, then n, so that the
// concurrent CTAs share a few A panels and a few W panels that stay in L2 (p.band = all m-groups
// gives plain m-fastest order). An m-tile past the last row reads zeros and stores nothing.
// Grouped (CL == 1): t numbers (group, n-tile, m-tile) with m fastest, so the m-tiles of one
// expert's W tile run side by side.
template <bool GROUPED, int CL>
__device__ __forceinline__ TileInfo decode_tile(int t, const GemmArgs& p, const int* s_tstart,
                                                const int* s_off, int crank)
{
    TileInfo ti;
    if constexpr (!GROUPED) {
        const int mgroups = (p.MT + CL - 1) / CL;
        const int per_band = p.band * p.NT;
        const int mb0 = (t / per_band) * p.band;             // first m-group of t's band
        const int bw = min(p.band, mgroups - mb0);           // m-groups in that band
        const int r = t - mb0 * p.NT;                        // item within the band
        const int mt = (mb0 + r % bw) * CL + crank;
        const int nt = r / bw;
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
        const int nt = local / mtg;
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

__device__ __forceinline__ uint64_t ld_shared_u64(uint32_t addr)
{
    uint64_t v;
    asm volatile("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v)
{
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// SiLU in FP32, g / (1 + e^-g), with the fast exponential and division intrinsics (a few FP32
// ulps; the accurate forms made the fused epilogue's tail 20% of the GEMM). For g below about
// -88 the exponential overflows to +inf and the result is -0.
__device__ __forceinline__ float silu(float g)
{
    return __fdividef(g, 1.0f + __expf(-g));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
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

__device__ __forceinline__ void st_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// QO: the output re-quantized to E4M3 in 1x128 tiles (codes to p.c, scales to p.h_s).
// DEFER: output tiles written by the store warp (dense BF16 output or QO).
template <bool GROUPED, bool OUT_F32, bool PAIR, bool RS, bool SW, bool QO = false,
          bool DEFER = false>
__global__ void __launch_bounds__(THREADS, 1)
fp8_blockscaled_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                            const __grid_constant__ CUtensorMap map_b,
                            const __grid_constant__ CUtensorMap map_c, const GemmArgs p)
{
    using L = Layout<GROUPED, PAIR, RS, SW>;
    static_assert(!SW || (GROUPED && !PAIR && !RS && !OUT_F32), "SwiGLU epilogue: grouped only");
    static_assert(!QO || (!GROUPED && !RS && !SW && !OUT_F32), "re-quantized output: dense only");
    constexpr int STAGES = L::STAGES;
    constexpr int CL = L::CL;
    // Output stores through the TMA engine (see the store below): the dense kernels with BF16
    // output and the row-scaled one. The plain dense kernel with FP32 output keeps 32-column
    // TMEM chunks and plain stores (with the bulk path it spilled and ran 23% slower).
    constexpr bool BULK_STORE = !GROUPED && !SW && !QO && (RS || !OUT_F32);
    // DEFER (dense BF16 output or QO, chosen by the host for long K loops and several tiles per
    // pair):
    // the epilogue stages a finished tile whole in shared memory and goes on to the next tile at
    // once; the store warp writes the staged tile to C meanwhile. (One warp needs ~2 us for a
    // tile: with short K loops it fell behind, and a pair's last tile waited for it.)
    constexpr bool DEFER_STORE = DEFER;
    static_assert(!DEFER || (PAIR && !GROUPED && !RS && !SW && !OUT_F32),
                  "store warp: dense, BF16 output or E4M3 codes (QO)");
    // the staged tile's element size, and its 32-row x 64-byte blocks per epilogue warp
    constexpr int OUT_ELEM = QO ? 1 : 2;
    constexpr int OUT_BLOCKS = 128 * OUT_ELEM / 64;
    // Odd-CTA epilogue warps release TMEM straight to the even CTA (2% faster than forwarding
    // through the odd CTA's MMA warp); the row-scaled epilogue keeps the forwarding, which costs
    // it no registers (the remote address spills there).
    constexpr bool DIRECT_RELEASE = PAIR && !RS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + (ALIGN_PAD - 1)) & ~static_cast<uint32_t>(ALIGN_PAD - 1);
    uint8_t* smem = smem_raw + (base - raw);

    const uint32_t sA = base + L::A_OFF;
    const uint32_t sB = base + L::B_OFF;
    const uint32_t bar0 = base + L::BAR_OFF;
    const uint32_t full0 = bar0;
    const uint32_t empty0 = bar0 + 8 * STAGES;
    const uint32_t tfull0 = bar0 + 16 * STAGES;
    const uint32_t tempty0 = tfull0 + 16;
    const uint32_t drain_bar = tempty0 + 16;
    const uint32_t sfull0 = drain_bar + 8;
    const uint32_t sempty0 = sfull0 + 8 * SCALE_SLOTS;
    const uint32_t ostaged = sempty0 + 8 * SCALE_SLOTS;   // DEFER_STORE only
    const uint32_t ofree = ostaged + 8;                   // DEFER_STORE only
    const uint32_t xch0 = ofree + 8;                      // SW only
    const uint32_t scl0 = base + L::SCL_OFF;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
    const uint32_t abort_addr = base + L::MISC_OFF + 4;   // shared word: a role gave up
    int* s_tstart = reinterpret_cast<int*>(smem + L::GROUP_OFF);   // grouped: [G+1]
    int* s_off = s_tstart + (p.G + 1);                               // grouped: [G+1]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long budget = p.budget;
    const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = (crank & 1u) == 0u;   // the even CTA of a pair issues the pair's MMAs
    const int cluster_id = blockIdx.x / CL;
    const int num_clusters = gridDim.x / CL;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(tfull0 + 8 * b, 1);
            // the local epilogue warps, plus (even CTA of a pair) the odd CTA's: its epilogue
            // warps' own remote arrives, or one forwarded arrive
            mbar_init(tempty0 + 8 * b,
                      NUM_EPI_WARPS + ((PAIR && leader) ? (DIRECT_RELEASE ? NUM_EPI_WARPS : 1) : 0));
        }
        mbar_init(drain_bar, 1);
        for (int i = 0; i < SCALE_SLOTS; i++) {
            mbar_init(sfull0 + 8 * i, 32);              // one cp.async completion per loader lane
            mbar_init(sempty0 + 8 * i, NUM_EPI_WARPS);
        }
        if constexpr (DEFER_STORE) {
            mbar_init(ostaged, NUM_EPI_WARPS);   // every epilogue warp has staged its rows
            mbar_init(ofree, 1);                 // the store warp has read the staged tile
        }
        if constexpr (SW) {
            for (int q = 0; q < 4; q++) mbar_init(xch0 + 8 * q, 2);   // the two warps of a quad
        }
        st_shared_volatile_u32(abort_addr, 0u);
        fence_mbar_init();
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
    }
    if (warp == MMA_WARP) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_holder), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
            tmem_relinquish();
        }
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
    if constexpr (PAIR) cluster_sync();   // the peer's barriers exist before anything targets them
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    int num_tiles = p.num_tiles;
    if constexpr (GROUPED) num_tiles = s_tstart[p.G];
    const int KB = p.KB;
    // The barriers the pair's MMA waits on live in the even CTA (rank crank & ~1).

    if (warp < EPI_WARP0) {
        regs_dec<REGS_CONTROL>();
        if (warp == PRODUCER_WARP) {
            // ---------------------------------------------------------------- TMA producer
            if (lane == 0) {
                const uint32_t full_lead0 = PAIR ? mapa_shared(full0, crank & ~1u) : full0;
                uint32_t it = 0;
                bool ok = true;
                for (int t = cluster_id; ok && t < num_tiles; t += num_clusters) {
                    const TileInfo ti =
                        decode_tile<GROUPED, CL>(t, p, s_tstart, s_off, static_cast<int>(crank));
                    for (int kb = 0; kb < KB; kb++, it++) {
                        const uint32_t s = it % STAGES;
                        const uint32_t ph = (it / STAGES) & 1u;
                        if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_addr, budget)) {
                            raise_error(p.err, abort_addr, DEV_TIMEOUT_PRODUCER);
                            ok = false;
                            break;
                        }
                        if constexpr (PAIR) {
                            // the even CTA's barrier counts the bytes of both CTAs
                            if (leader) mbar_arrive_expect_tx(full0 + 8 * s, CL * L::STAGE);
                            tma_load_2d_pair(sA + s * A_BYTES, &map_a, full_lead0 + 8 * s, kb * BK,
                                             static_cast<int32_t>(ti.row0));
                            tma_load_2d_pair(sB + s * L::B_PART, &map_b, full_lead0 + 8 * s,
                                             kb * BK,
                                             static_cast<int32_t>(ti.wrow0 + crank * (BN / CL)));
                        } else {
                            mbar_arrive_expect_tx(full0 + 8 * s, L::STAGE);
                            tma_load_2d(sA + s * A_BYTES, &map_a, full0 + 8 * s, kb * BK,
                                        static_cast<int32_t>(ti.row0));
                            tma_load_2d(sB + s * L::B_PART, &map_b, full0 + 8 * s, kb * BK,
                                        static_cast<int32_t>(ti.wrow0));
                        }
                    }
                }
                if ((!ok || ld_shared_volatile_u32(abort_addr) != 0) && leader) {
                    // After an abort the MMA side may never consume what is in flight: wait for
                    // the last copy issued into every stage before the CTA may exit.
                    const uint32_t first = it > STAGES ? it - STAGES : 0;
                    for (uint32_t i = first; i < it; i++)
                        if (!mbar_wait(full0 + 8 * (i % STAGES), (i / STAGES) & 1u, 0u, budget))
                            atomicCAS(p.err, 0, DEV_TIMEOUT_DRAIN);
                }
            }
        } else if (warp == MMA_WARP) {
            // ---------------------------------------------------------------- MMA issuer
            if (lane == 0 && leader) {
                constexpr uint32_t IDESC = idesc_e4m3_f32(BM * CL, BN);
                constexpr uint16_t PAIR_MASK = 0x3;
                uint32_t it = 0, j = 0;
                bool ok = true, issued = false;
                for (int t = cluster_id; ok && t < num_tiles; t += num_clusters) {
                    for (int kb = 0; kb < KB; kb++, it++, j++) {
                        const uint32_t b = j % TMEM_BUFS;
                        const uint32_t pb = (j / TMEM_BUFS) & 1u;
                        const bool freed = mbar_wait(tempty0 + 8 * b, pb ^ 1u, abort_addr, budget);
                        if (!freed) {
                            raise_error(p.err, abort_addr, DEV_TIMEOUT_MMA_TMEM);
                            ok = false;
                            break;
                        }
                        const uint32_t s = it % STAGES;
                        const uint32_t ph = (it / STAGES) & 1u;
                        const bool filled = mbar_wait(full0 + 8 * s, ph, abort_addr, budget);
                        if (!filled) {
                            raise_error(p.err, abort_addr, DEV_TIMEOUT_MMA_FULL);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t da = desc_kmajor_sw128(sA + s * A_BYTES);
                        const uint64_t db = desc_kmajor_sw128(sB + s * L::B_PART);
                        const uint32_t d_tmem = tmem_base + b * BN;
#pragma unroll
                        for (int k = 0; k < BK / 32; k++) {   // +32 bytes of K = +2 in the address field
                            if constexpr (PAIR)
                                mma_e4m3_pair(d_tmem, da + 2 * k, db + 2 * k, IDESC, k > 0 ? 1u : 0u);
                            else
                                mma_e4m3(d_tmem, da + 2 * k, db + 2 * k, IDESC, k > 0 ? 1u : 0u);
                        }
                        if constexpr (PAIR) {
                            mma_commit_pair_multicast(empty0 + 8 * s, PAIR_MASK);
                            mma_commit_pair_multicast(tfull0 + 8 * b, PAIR_MASK);
                        } else {
                            mma_commit(empty0 + 8 * s);
                            mma_commit(tfull0 + 8 * b);
                        }
                        issued = true;
                    }
                }
                if (issued) {
                    // Every MMA must have finished before TMEM is released.
                    if constexpr (PAIR)
                        mma_commit_pair_multicast(drain_bar, static_cast<uint16_t>(1u << crank));
                    else
                        mma_commit(drain_bar);
                    if (!mbar_wait(drain_bar, 0, 0u, budget)) atomicCAS(p.err, 0, DEV_TIMEOUT_DRAIN);
                }
            } else if (PAIR && !DIRECT_RELEASE && !leader && lane == 0) {
                // Odd CTA of a pair (variants whose epilogue has no register to spare for the
                // remote release): forward the release of each TMEM accumulator by this CTA's
                // epilogue (its local tempty barrier) to the even CTA, whose MMA waits for both.
                const uint32_t peer_tempty0 = mapa_shared(tempty0, crank & ~1u);
                uint32_t j = 0;
                bool ok = true;
                for (int t = cluster_id; ok && t < num_tiles; t += num_clusters) {
                    for (int kb = 0; kb < KB; kb++, j++) {
                        const uint32_t b = j % TMEM_BUFS;
                        if (!mbar_wait(tempty0 + 8 * b, (j / TMEM_BUFS) & 1u, abort_addr, budget)) {
                            raise_error(p.err, abort_addr, DEV_TIMEOUT_MMA_TMEM);
                            ok = false;
                            break;
                        }
                        mbar_arrive_cluster(peer_tempty0 + 8 * b);
                    }
                }
            }
            __syncwarp();
        } else if (warp == SCALE_WARP) {
            // ---------------------------------------------------------------- scale loader
            // Slot it % SCALE_SLOTS receives the K block's 128 activation scales (rows of this
            // CTA's tile; zero past the last row) and the scales of the tile's two weight blocks,
            // by asynchronous copies whose completion arrives on sfull. The epilogue frees it.
            uint32_t it = 0;
            bool ok = true;
            const float* zero_src = p.a_s;   // any valid address; zero-filled copies read nothing
            for (int t = cluster_id; ok && t < num_tiles; t += num_clusters) {
                const TileInfo ti =
                    decode_tile<GROUPED, CL>(t, p, s_tstart, s_off, static_cast<int>(crank));
                bool rv[4];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int64_t row = ti.row0 + lane + 32 * q;
                    rv[q] = row >= 0 && row < ti.row_end;
                }
                const int nb = ti.n0 / 128 + lane;           // lanes 0, 1: the two weight blocks
                const bool wv = lane < 2 && nb < p.NB;
                const float* w_base =
                    p.w_s + (static_cast<int64_t>(ti.g) * p.NB + (wv ? nb : 0)) * KB;
                bool cv[RS ? 8 : 1];                         // RS: B rows n0 + lane + 32 q exist
#pragma unroll
                for (int q = 0; q < (RS ? 8 : 1); q++) cv[q] = ti.n0 + lane + 32 * q < p.N;
                for (int kb = 0; kb < KB; kb++, it++) {
                    const uint32_t slot = it % SCALE_SLOTS;
                    const uint32_t ph = (it / SCALE_SLOTS) & 1u;
                    const bool got = mbar_wait(sempty0 + 8 * slot, ph ^ 1u, abort_addr, budget);
                    if (!__all_sync(0xffffffffu, got)) {
                        if (lane == 0) raise_error(p.err, abort_addr, DEV_TIMEOUT_SCALES);
                        ok = false;
                        break;
                    }
                    const uint32_t dst = scl0 + slot * L::SLOT;
                    const float* a_row = p.a_s + static_cast<int64_t>(kb) * p.rows + ti.row0;
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        cp_async_4(dst + (lane + 32 * q) * 4,
                                   rv[q] ? a_row + lane + 32 * q : zero_src, rv[q] ? 4u : 0u);
                    if constexpr (RS) {
                        // the 256 B-row scales of this K block: b_s[kb][n0 .. n0 + 255]
                        const float* b_row = p.w_s + static_cast<int64_t>(kb) * p.N + ti.n0;
#pragma unroll
                        for (int q = 0; q < 8; q++)
                            cp_async_4(dst + 512 + (lane + 32 * q) * 4,
                                       cv[q] ? b_row + lane + 32 * q : zero_src, cv[q] ? 4u : 0u);
                    } else if (lane < 2) {
                        cp_async_4(dst + 512 + lane * 4, wv ? w_base + kb : zero_src, wv ? 4u : 0u);
                    }
                    cp_async_mbar_arrive(sfull0 + 8 * slot);
                }
            }
            // Copies still in flight complete on their own; wait for them before the CTA exits.
            if (it > 0) {
                const uint32_t first = it > SCALE_SLOTS ? it - SCALE_SLOTS : 0;
                for (uint32_t i = first; i < it; i++)
                    if (!mbar_wait(sfull0 + 8 * (i % SCALE_SLOTS), (i / SCALE_SLOTS) & 1u, 0u,
                                   budget))
                        atomicCAS(p.err, 0, DEV_TIMEOUT_DRAIN);
            }
        } else if (DEFER_STORE && warp == STORE_WARP) {
            // ---------------------------------------------------------------- store warp
            // Each staged output tile goes to C, 8 rows of 64 contiguous bytes per store
            // instruction (row- and column-predicated), while the epilogue works on the next
            // tile; then the staging buffer is handed back.
            uint32_t n = 0;
            const int ch = lane & 3;
            for (int t = cluster_id; t < num_tiles; t += num_clusters, n++) {
                const bool got = mbar_wait(ostaged, n & 1u, abort_addr, budget);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0) raise_error(p.err, abort_addr, DEV_TIMEOUT_EPILOGUE);
                    break;
                }
                const TileInfo ts =
                    decode_tile<GROUPED, CL>(t, p, s_tstart, s_off, static_cast<int>(crank));
#pragma unroll 1
                for (int w = 0; w < NUM_EPI_WARPS; w++) {
                    // epilogue warp EPI_WARP0 + w: TMEM lane quarter w % 4, column half w / 4
                    const uint32_t buf = base + L::STG_OFF + w * 4 * STG_WARP_BYTES;
                    const int64_t wrow0 = ts.row0 + (w & 3) * 32;
                    const int col0 = ts.n0 + (w >> 2) * 128;
#pragma unroll
                    for (int g = 0; g < OUT_BLOCKS; g++) {
                        const int gcol = col0 + g * (64 / OUT_ELEM) + ch * (16 / OUT_ELEM);
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const int rr = i * 8 + (lane >> 2);
                            const uint4 v = ld_shared_v4(buf + g * STG_WARP_BYTES + rr * 64 +
                                                         ((ch ^ ((rr >> 1) & 3)) * 16));
                            const int64_t grow = wrow0 + rr;
                            if (grow < ts.row_end && gcol < p.N)
                                st_v4(static_cast<uint8_t*>(p.c) + (grow * p.ldc + gcol) * OUT_ELEM,
                                      v.x, v.y, v.z, v.w);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(ofree);
            }
        }
    } else {
        regs_inc<REGS_EPILOGUE>();
        // ---------------------------------------------------------------- epilogue
        const int quad = warp & 3;                   // TMEM lanes 32*quad .. 32*quad + 31
        const int half = (warp - EPI_WARP0) >> 2;    // columns 128*half .. 128*half + 127 (SW:
                                                     // gate 64*half.. + 63 and up 128 + 64*half..)
        const int r = quad * 32 + lane;              // row within the tile
        const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
        // the even CTA's tempty barriers as cluster addresses (QO's form of the remote release)
        const uint32_t release0 = PAIR ? mapa_shared(tempty0, crank & ~1u) : tempty0;
        uint32_t j = 0;
        uint64_t acc[64];   // 128 FP32 accumulators as packed pairs (columns 2i, 2i + 1)
        uint32_t tile_n = 0;   // tiles finished by this CTA (SW: parity of the exchange buffers)
        // DEFER_STORE: this warp's part of the staged output tile (32 rows x 128 columns)
        const uint32_t d_buf = base + L::STG_OFF + (warp - EPI_WARP0) * 4 * STG_WARP_BYTES;

        for (int t = cluster_id; t < num_tiles; t += num_clusters, tile_n++) {
            const int ncol0 =
                decode_tile<GROUPED, CL>(t, p, s_tstart, s_off, static_cast<int>(crank)).n0 +
                half * 128;
#pragma unroll
            for (int i = 0; i < 64; i++) acc[i] = 0ull;

            bool ok = true;
            for (int kb = 0; kb < KB; kb++, j++) {
                // This K block's scales from the scale ring (filled ahead by the loader warp).
                const uint32_t slot = j % SCALE_SLOTS;
                const bool sgot =
                    mbar_wait(sfull0 + 8 * slot, (j / SCALE_SLOTS) & 1u, abort_addr, budget);
                if (!__all_sync(0xffffffffu, sgot)) {
                    if (lane == 0) raise_error(p.err, abort_addr, DEV_TIMEOUT_EPILOGUE);
                    ok = false;
                    break;
                }
                const uint32_t sl = scl0 + slot * L::SLOT;
                // Block-scaled B: one product s_a[row] * s_w[block] per K block. RS: s_a[row]
                // here, times s_b[column] per column pair below (B-row scales stay in the slot
                // until the promotion is done).
                // SW: the gate half of the tile (W block 2 nt) and the up half (block 2 nt + 1).
                const float sc = RS ? ld_shared_f32(sl + r * 4)
                                    : __fmul_rn(ld_shared_f32(sl + r * 4),
                                                ld_shared_f32(sl + 512 + (SW ? 0 : half) * 4));
                const float sc_up =
                    SW ? __fmul_rn(ld_shared_f32(sl + r * 4), ld_shared_f32(sl + 516)) : sc;
                const uint32_t sb = sl + 512 + half * 128 * 4;   // RS: s_b of this half's columns
                if constexpr (!RS) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sempty0 + 8 * slot);
                }

                const uint32_t b = j % TMEM_BUFS;
                const uint32_t pb = (j / TMEM_BUFS) & 1u;
                const bool got = mbar_wait(tfull0 + 8 * b, pb, abort_addr, budget);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0) raise_error(p.err, abort_addr, DEV_TIMEOUT_EPILOGUE);
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Four 32-column chunks; the TMEM load of chunk c+1 is in flight while chunk c
                // is promoted (two register buffers of 16 packed pairs).
                const uint32_t taddr = tmem_base + t_lane + b * BN + half * (SW ? 64 : 128);
                const uint64_t sc2 = f32x2_splat(sc);
                const uint64_t sc2b = f32x2_splat(sc_up);        // SW: the up columns
                if constexpr (RS) {
                    // Per-column scales, eight 16-column chunks: acc = fma(P * s_b[n], s_a[m], acc)
                    // (the product P * s_b depends on the TMEM data, so it is formed only when
                    // the chunk has arrived instead of being computed ahead into registers).
                    uint64_t u0[8], u1[8];
                    tmem_ld_16cols(taddr, u0);
#pragma unroll
                    for (int c = 0; c < 8; c += 2) {
                        __syncwarp();   // with the form above, keeps the epilogue within its registers
                        tmem_wait_ld(u0);
                        tmem_ld_16cols(taddr + 16 * (c + 1), u1);
#pragma unroll
                        for (int i = 0; i < 8; i++)
                            ffma2(acc[8 * c + i], fmul2(u0[i], ld_shared_u64(sb + 64 * c + 8 * i)),
                                  sc2);
                        tmem_wait_ld(u1);
                        if (c + 2 < 8) tmem_ld_16cols(taddr + 16 * (c + 2), u0);
#pragma unroll
                        for (int i = 0; i < 8; i++)
                            ffma2(acc[8 * (c + 1) + i],
                                  fmul2(u1[i], ld_shared_u64(sb + 64 * (c + 1) + 8 * i)), sc2);
                    }
                } else if constexpr (SW || QO || (BULK_STORE && !DEFER_STORE)) {
                    // SW: gate columns 64 half .. + 63 into acc[0..31] (scale s_a * s_w[gate
                    // block]), up columns 128 + 64 half .. + 63 into acc[32..63] (s_a * s_w[up
                    // block]); otherwise the usual 128 columns, one scale. 16-column chunks
                    // leave registers for the tail that follows the K loop (the fused tails, and
                    // the bulk output stores; the store-warp variant's short tail fits beside
                    // 32-column chunks, 0.5-1% faster).
                    auto col = [](int c) -> uint32_t {
                        return (SW && c >= 4) ? 128 + 16 * (c - 4) : 16 * c;
                    };
                    uint64_t u0[8], u1[8];
                    tmem_ld_16cols(taddr, u0);
#pragma unroll
                    for (int c = 0; c < 8; c += 2) {
                        const uint32_t col1 = col(c + 1);
                        tmem_wait_ld(u0);
                        tmem_ld_16cols(taddr + col1, u1);
#pragma unroll
                        for (int i = 0; i < 8; i++) ffma2(acc[8 * c + i], u0[i], c < 4 ? sc2 : sc2b);
                        tmem_wait_ld(u1);
                        if (c + 2 < 8) tmem_ld_16cols(taddr + col(c + 2), u0);
#pragma unroll
                        for (int i = 0; i < 8; i++)
                            ffma2(acc[8 * (c + 1) + i], u1[i], c + 1 < 4 ? sc2 : sc2b);
                    }
                } else {
                    // four 32-column chunks
                    uint64_t v0[16], v1[16];
                    tmem_ld_32cols(taddr, v0);
                    tmem_wait_ld(v0);
                    tmem_ld_32cols(taddr + 32, v1);
#pragma unroll
                    for (int i = 0; i < 16; i++) ffma2(acc[i], v0[i], sc2);
                    tmem_wait_ld(v1);
                    tmem_ld_32cols(taddr + 64, v0);
#pragma unroll
                    for (int i = 0; i < 16; i++) ffma2(acc[16 + i], v1[i], sc2);
                    tmem_wait_ld(v0);
                    tmem_ld_32cols(taddr + 96, v1);
#pragma unroll
                    for (int i = 0; i < 16; i++) ffma2(acc[32 + i], v0[i], sc2);
                    tmem_wait_ld(v1);
#pragma unroll
                    for (int i = 0; i < 16; i++) ffma2(acc[48 + i], v1[i], sc2);
                }
                tc_fence_before();
                __syncwarp();
                if constexpr (RS) {
                    if (lane == 0) mbar_arrive(sempty0 + 8 * slot);
                }
                // (test hook: one epilogue warp can be told to skip one release, see GemmArgs)
                // A pair's MMAs write both CTAs' TMEM: the odd CTA's warps release their half of
                // the buffer on the even CTA's barrier with a plain remote arrive (the TMEM reads
                // are already ordered by tcgen05.wait::ld and the fence above).
                if (lane == 0 && !(warp == EPI_WARP0 && static_cast<int>(j) == p.fault_skip_release)) {
                    // (the two forms of the remote arrive are the ones that fit each variant's
                    // registers without spilling)
                    if constexpr (DIRECT_RELEASE && QO)
                        mbar_arrive_cluster(release0 + 8 * b);
                    else if (DIRECT_RELEASE && !leader)
                        mbar_arrive_cluster(mapa_shared(tempty0 + 8 * b, crank & ~1u));
                    else
                        mbar_arrive(tempty0 + 8 * b);
                }

            }
            if (!ok) break;

            if constexpr (SW) {
                // h = silu(g) * u for this thread's 64 channels (g in acc[0..31], u in
                // acc[32..63]), then the 1x128 tile of h: its amax combines this warp's 64
                // channels with the partner warp's (same rows, other half), exchanged through
                // shared memory; then scale, codes, and a staged store of 64 codes per row.
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    const float h0 = __fmul_rn(silu(f32x2_lo(acc[i])), f32x2_lo(acc[32 + i]));
                    const float h1 = __fmul_rn(silu(f32x2_hi(acc[i])), f32x2_hi(acc[32 + i]));
                    acc[i] = f32x2_pack(h0, h1);
                    amax = fmaxf(amax, fmaxf(fabsf(h0), fabsf(h1)));
                }
                const uint32_t xbuf = base + L::XCH_OFF + (tile_n & 1u) * 1024;
                st_shared_f32(xbuf + half * 512 + r * 4, amax);
                __syncwarp();
                if (lane == 0) mbar_arrive(xch0 + 8 * quad);
                const bool xok = mbar_wait(xch0 + 8 * quad, tile_n & 1u, abort_addr, budget);
                if (!__all_sync(0xffffffffu, xok)) {
                    if (lane == 0) raise_error(p.err, abort_addr, DEV_TIMEOUT_EPILOGUE);
                    break;
                }
                amax = fmaxf(amax, ld_shared_f32(xbuf + (half ^ 1) * 512 + r * 4));
                const TileScale tsc = tile_scale(amax);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const uint32_t lo = cvt_e4m3x2(tile_scaled(f32x2_lo(acc[2 * i]), tsc),
                                                   tile_scaled(f32x2_hi(acc[2 * i]), tsc));
                    const uint32_t hi = cvt_e4m3x2(tile_scaled(f32x2_lo(acc[2 * i + 1]), tsc),
                                                   tile_scaled(f32x2_hi(acc[2 * i + 1]), tsc));
                    w[i] = tsc.zero ? 0u : (lo | (hi << 16));
                }
                const TileInfo ts =
                    decode_tile<GROUPED, CL>(t, p, s_tstart, s_off, static_cast<int>(crank));
                const int64_t grow_own = ts.row0 + r;
                const int ob = ts.n0 / BN;                       // 1x128 output tile index
                if (half == 0 && grow_own < ts.row_end)
                    p.h_s[static_cast<int64_t>(ob) * p.rows + grow_own] = tsc.s;
                // 32 rows x 64 code bytes of this warp, staged as in the store below
                const uint32_t stg = base + L::STG_OFF + (warp - EPI_WARP0) * STG_WARP_BYTES;
#pragma unroll
                for (int jc = 0; jc < 4; jc++)
                    st_shared_v4(stg + lane * 64 + (((jc + (lane >> 1)) & 3) * 16),
                                 make_uint4(w[4 * jc], w[4 * jc + 1], w[4 * jc + 2], w[4 * jc + 3]));
                __syncwarp();
                const int ch = lane & 3;
                const int64_t gcol = static_cast<int64_t>(ob) * 128 + half * 64 + ch * 16;
                const int64_t wrow0 = ts.row0 + quad * 32;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int rr = i * 8 + (lane >> 2);
                    const uint4 v = ld_shared_v4(stg + rr * 64 + (((ch + (rr >> 1)) & 3) * 16));
                    const int64_t grow = wrow0 + rr;
                    if (grow < ts.row_end)
                        st_v4(static_cast<uint8_t*>(p.c) + grow * p.ldc + gcol, v.x, v.y, v.z, v.w);
                }
                __syncwarp();
                continue;
            }

            if constexpr (QO) {
                // The output re-quantized in 1x128 tiles, the layout the next GEMM reads for its
                // A operand: this thread's 128 columns of its row are one tile, so its amax,
                // scale (the quantizers' tile_scale) and codes need nothing from other threads.
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 64; i++)
                    amax = fmaxf(amax, fmaxf(fabsf(f32x2_lo(acc[i])), fabsf(f32x2_hi(acc[i]))));
                const TileScale tsc = tile_scale(amax);
                const TileInfo ts =
                    decode_tile<GROUPED, CL>(t, p, s_tstart, s_off, static_cast<int>(crank));
                const int col0 = ts.n0 + half * 128;            // first column of the tile
                const int64_t grow_own = ts.row0 + r;
                if (grow_own < ts.row_end && col0 < p.N)
                    p.h_s[static_cast<int64_t>(col0 / 128) * p.rows + grow_own] = tsc.s;
                if constexpr (DEFER_STORE) {
                    // the store warp writes the codes: stage them as the BF16 path does, in two
                    // 32-row x 64-byte blocks, once the store warp has read the previous tile
                    const bool freed = mbar_wait(ofree, (tile_n & 1u) ^ 1u, abort_addr, budget);
                    if (!__all_sync(0xffffffffu, freed)) {
                        if (lane == 0) raise_error(p.err, abort_addr, DEV_TIMEOUT_EPILOGUE);
                        break;
                    }
#pragma unroll
                    for (int g = 0; g < 2; g++) {
#pragma unroll
                        for (int jc = 0; jc < 4; jc++) {
                            uint32_t w4[4];
#pragma unroll
                            for (int e = 0; e < 4; e++) {
                                const int q = g * 32 + jc * 8 + 2 * e;
                                const uint32_t lo =
                                    cvt_e4m3x2(tile_scaled(f32x2_lo(acc[q]), tsc),
                                               tile_scaled(f32x2_hi(acc[q]), tsc));
                                const uint32_t hi =
                                    cvt_e4m3x2(tile_scaled(f32x2_lo(acc[q + 1]), tsc),
                                               tile_scaled(f32x2_hi(acc[q + 1]), tsc));
                                w4[e] = tsc.zero ? 0u : (lo | (hi << 16));
                            }
                            st_shared_v4(d_buf + g * STG_WARP_BYTES + lane * 64 +
                                             ((jc ^ ((lane >> 1) & 3)) * 16),
                                         make_uint4(w4[0], w4[1], w4[2], w4[3]));
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ostaged);
                    continue;
                }
                const uint32_t stg = base + L::STG_OFF + (warp - EPI_WARP0) * STG_WARP_BYTES;
                const int64_t wrow0 = ts.row0 + quad * 32;
#pragma unroll
                for (int g = 0; g < 2; g++) {                    // 64 codes (64 B) per round
#pragma unroll
                    for (int jc = 0; jc < 4; jc++) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int q = g * 32 + jc * 8 + 2 * e;
                            const uint32_t lo = cvt_e4m3x2(tile_scaled(f32x2_lo(acc[q]), tsc),
                                                           tile_scaled(f32x2_hi(acc[q]), tsc));
                            const uint32_t hi = cvt_e4m3x2(tile_scaled(f32x2_lo(acc[q + 1]), tsc),
                                                           tile_scaled(f32x2_hi(acc[q + 1]), tsc));
                            w4[e] = tsc.zero ? 0u : (lo | (hi << 16));
                        }
                        st_shared_v4(stg + lane * 64 + (((jc + (lane >> 1)) & 3) * 16),
                                     make_uint4(w4[0], w4[1], w4[2], w4[3]));
                    }
                    __syncwarp();
                    const int ch = lane & 3;
                    const int gcol = col0 + g * 64 + ch * 16;
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int rr = i * 8 + (lane >> 2);
                        const uint4 v = ld_shared_v4(stg + rr * 64 + (((ch + (rr >> 1)) & 3) * 16));
                        const int64_t grow = wrow0 + rr;
                        if (grow < ts.row_end && gcol < p.N)
                            st_v4(static_cast<uint8_t*>(p.c) + grow * p.ldc + gcol, v.x, v.y, v.z, v.w);
                    }
                    __syncwarp();
                }
                continue;
            }

            if constexpr (DEFER_STORE) {
                // Once the store warp has read the previous staged tile, this warp stages its 32
                // rows x 128 columns in four 2 KB blocks of 32 rows x 64 B (chunk j of row r at
                // position j ^ ((r / 2) % 4), conflict-free both ways) and goes on to the next
                // tile; the store warp writes them out meanwhile.
                const bool freed = mbar_wait(ofree, (tile_n & 1u) ^ 1u, abort_addr, budget);
                if (!__all_sync(0xffffffffu, freed)) {
                    if (lane == 0) raise_error(p.err, abort_addr, DEV_TIMEOUT_EPILOGUE);
                    break;
                }
#pragma unroll
                for (int g = 0; g < 4; g++) {
#pragma unroll
                    for (int jc = 0; jc < 4; jc++) {
                        const int q = g * 16 + jc * 4;
                        const uint4 v =
                            make_uint4(pack_bf16x2(f32x2_lo(acc[q]), f32x2_hi(acc[q])),
                                       pack_bf16x2(f32x2_lo(acc[q + 1]), f32x2_hi(acc[q + 1])),
                                       pack_bf16x2(f32x2_lo(acc[q + 2]), f32x2_hi(acc[q + 2])),
                                       pack_bf16x2(f32x2_lo(acc[q + 3]), f32x2_hi(acc[q + 3])));
                        st_shared_v4(d_buf + g * STG_WARP_BYTES + lane * 64 +
                                         ((jc ^ ((lane >> 1) & 3)) * 16),
                                     v);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(ostaged);
                continue;
            }

            // Store: this warp's 32 rows go out 64 bytes of each row at a time, staged in a 2 KB
            // shared buffer: chunk j (16 B) of row r at position j ^ ((r / 2) % 4), which keeps
            // the row-wise writes here and the column-wise reads below free of bank conflicts.
            // BULK_STORE: the staged buffer is the output map's box (that position is its 64-byte
            // swizzle); one lane hands it to the TMA engine and the warp goes on, waiting only
            // for the engine to have read the buffer before refilling it, so the global writes
            // overlap the next tile's K loop. Otherwise plain row-predicated stores, 8 rows of 64
            // bytes per instruction: grouped (rows past a group's end belong to the next group's
            // output, which the map cannot clip; bulk stores also measured 3-4% slower on the
            // HBM-bound grouped shapes) and dense FP32.
            {
                constexpr int ELEM = OUT_F32 ? 4 : 2;
                constexpr int GCOLS = 64 / ELEM;             // columns per 64-byte staged row
                const TileInfo ts =
                    decode_tile<GROUPED, CL>(t, p, s_tstart, s_off, static_cast<int>(crank));
                const uint32_t stg = base + L::STG_OFF + (warp - EPI_WARP0) * STG_WARP_BYTES;
                const int64_t wrow0 = ts.row0 + quad * 32;   // first row of this warp
                // (rows past M are outside the output map and not written)
                constexpr bool bulk = BULK_STORE;
#pragma unroll
                for (int g = 0; g < 128 / GCOLS; g++) {
                    if (bulk && lane == 0) bulk_wait_group_read<0>();   // its last box was read
                    __syncwarp();
#pragma unroll
                    for (int jc = 0; jc < 4; jc++) {
                        uint4 v;
                        if constexpr (OUT_F32) {
                            const uint64_t p0 = acc[g * 8 + jc * 2], p1 = acc[g * 8 + jc * 2 + 1];
                            v = make_uint4(static_cast<uint32_t>(p0), static_cast<uint32_t>(p0 >> 32),
                                           static_cast<uint32_t>(p1), static_cast<uint32_t>(p1 >> 32));
                        } else {
                            const int q = g * 16 + jc * 4;
                            v = make_uint4(pack_bf16x2(f32x2_lo(acc[q]), f32x2_hi(acc[q])),
                                           pack_bf16x2(f32x2_lo(acc[q + 1]), f32x2_hi(acc[q + 1])),
                                           pack_bf16x2(f32x2_lo(acc[q + 2]), f32x2_hi(acc[q + 2])),
                                           pack_bf16x2(f32x2_lo(acc[q + 3]), f32x2_hi(acc[q + 3])));
                        }
                        st_shared_v4(stg + lane * 64 + ((jc ^ ((lane >> 1) & 3)) * 16), v);
                    }
                    const int gcol0 = ncol0 + g * GCOLS;
                    if (bulk) {
                        fence_proxy_async_smem();            // the box is visible to the engine
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&map_c, stg, gcol0, static_cast<int32_t>(wrow0));
                            bulk_commit_group();
                        }
                    } else {
                        __syncwarp();
                        const int ch = lane & 3;
                        const int gcol = gcol0 + ch * (16 / ELEM);
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const int rr = i * 8 + (lane >> 2);
                            const uint4 v = ld_shared_v4(stg + rr * 64 + ((ch ^ ((rr >> 1) & 3)) * 16));
                            const int64_t grow = wrow0 + rr;
                            if (grow >= 0 && grow < ts.row_end && gcol < p.N)
                                st_v4(static_cast<uint8_t*>(p.c) + (grow * p.ldc + gcol) * ELEM, v.x,
                                      v.y, v.z, v.w);
                        }
                        __syncwarp();
                    }
                }
            }
        }
        // every output box this warp handed to the TMA engine has been written before the
        // CTA may finish
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();   // both CTAs are done with TMEM and the peer's barriers
    tc_fence_after();
    if (warp == MMA_WARP) {
        __syncwarp();
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if constexpr (PAIR) cluster_sync();   // no CTA leaves while its peer still deallocates
}

template <bool GROUPED, bool OUT_F32, bool PAIR, bool RS, bool SW = false, bool QO = false,
          bool DEFER = false>
cudaError_t launch_one(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                       const GemmArgs& args, int max_ctas, cudaStream_t stream)
{
    constexpr int CL = PAIR ? 2 : 1;
    auto kern = fp8_blockscaled_gemm_kernel<GROUPED, OUT_F32, PAIR, RS, SW, QO, DEFER>;
    const size_t smem = gemm_smem_bytes(
        SW ? GemmKind::GROUPED_SWIGLU
           : (RS ? GemmKind::ROW_SCALED : (GROUPED ? GemmKind::GROUPED : GemmKind::DENSE)),
        args.G);   // (the re-quantized output uses the dense layout)
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Persistent grid: as many clusters as fit at once (one CTA per SM), at most one per item.
    int clusters = max_ctas / CL;
    if (CL > 1) {
        cfg.gridDim = dim3(static_cast<unsigned>(clusters * CL));
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess) {
            cudaGetLastError();   // not fatal: keep one cluster per SM pair
            active = 0;
        }
        if (active > 0 && active < clusters) clusters = active;
    }
    if (!GROUPED && args.num_tiles < clusters) clusters = args.num_tiles;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * CL));
    e = cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

size_t gemm_smem_bytes(GemmKind kind, int G)
{
    constexpr bool DENSE_PAIR = GEMM_DENSE_CLUSTER == 2;
    const size_t group_table = 2 * static_cast<size_t>(G + 1) * sizeof(int);
    switch (kind) {
    case GemmKind::ROW_SCALED:
        return static_cast<size_t>(Layout<false, DENSE_PAIR, true>::GROUP_OFF) + ALIGN_PAD;
    case GemmKind::GROUPED:
        return static_cast<size_t>(Layout<true, false, false>::GROUP_OFF) + ALIGN_PAD + group_table;
    case GemmKind::GROUPED_SWIGLU:
        return static_cast<size_t>(Layout<true, false, false, true>::GROUP_OFF) + ALIGN_PAD +
               group_table;
    case GemmKind::DENSE:
    case GemmKind::DENSE_QUANT:
    default:
        return static_cast<size_t>(Layout<false, DENSE_PAIR, false>::GROUP_OFF) + ALIGN_PAD;
    }
}

int gemm_cluster_size(bool grouped) { return grouped ? 1 : GEMM_DENSE_CLUSTER; }

// Dense tile order. The concurrent clusters of one wave read, over the whole K loop, the A
// panels (cluster rows x K bytes) of the m-groups they cover and the W panels (BN x K bytes) of
// the n-tiles they cover; the next wave finds a panel in L2 only if the wave's panels fit there.
// Plain m-fastest order keeps all m-groups in every wave, which is best while that fits (all of
// A is read once). Otherwise bands of about sqrt(clusters) m-groups make a wave's panels as few
// as possible: each band's A panels are read once, the W panels once per band.
int gemm_band(int mgroups, int NT, int64_t K, int clusters)
{
    constexpr double L2_BUDGET = 48.0 * 1024 * 1024;   // of the 126 MB L2, for one wave's panels
    const double a_panel = static_cast<double>(GEMM_DENSE_CLUSTER * GEMM_BM) * K;
    const double b_panel = static_cast<double>(GEMM_BN) * K;
    const int P = clusters > 0 ? clusters : 1;
    const int mw = mgroups < P ? mgroups : P;
    const int nw = (P + mgroups - 1) / mgroups;
    if (mw * a_panel + (nw < NT ? nw : NT) * b_panel <= L2_BUDGET) return mgroups > 0 ? mgroups : 1;
    int b = 1;
    while ((b + 1) * (b + 1) * a_panel <= P * b_panel) b++;   // b ~ sqrt(P * b_panel / a_panel)
    return b < mgroups ? b : mgroups;
}

cudaError_t launch_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b,
                        const CUtensorMap& map_c, const GemmArgs& args, GemmKind kind,
                        bool out_f32, int max_ctas, cudaStream_t stream, bool store_warp)
{
    constexpr bool DP = GEMM_DENSE_CLUSTER == 2;
    switch (kind) {
    case GemmKind::GROUPED:
        return out_f32 ? launch_one<true, true, false, false>(map_a, map_b, map_c, args, max_ctas, stream)
                       : launch_one<true, false, false, false>(map_a, map_b, map_c, args, max_ctas, stream);
    case GemmKind::GROUPED_SWIGLU:
        return launch_one<true, false, false, false, true>(map_a, map_b, map_c, args, max_ctas, stream);
    case GemmKind::DENSE_QUANT:
        if (store_warp)
            return launch_one<false, false, DP, false, false, true, true>(map_a, map_b, map_c, args,
                                                                          max_ctas, stream);
        return launch_one<false, false, DP, false, false, true>(map_a, map_b, map_c, args, max_ctas,
                                                                stream);
    case GemmKind::ROW_SCALED:
        return out_f32 ? launch_one<false, true, DP, true>(map_a, map_b, map_c, args, max_ctas, stream)
                       : launch_one<false, false, DP, true>(map_a, map_b, map_c, args, max_ctas, stream);
    case GemmKind::DENSE:
    default:
        if (out_f32)
            return launch_one<false, true, DP, false>(map_a, map_b, map_c, args, max_ctas, stream);
        if (store_warp)
            return launch_one<false, false, DP, false, false, false, true>(map_a, map_b, map_c, args,
                                                                          max_ctas, stream);
        return launch_one<false, false, DP, false>(map_a, map_b, map_c, args, max_ctas, stream);
    }
}

}  // namespace fp8bs
