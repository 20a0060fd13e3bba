// internal.h -- launchers shared between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fp8bs.h"

namespace fp8bs {

constexpr int QUANT_THREADS = 256;

// GEMM tiling: one CTA computes a 128 x GEMM_BN tile of C; each pipeline stage holds one
// 128-wide K block (the quantization block) of A and W.
constexpr int GEMM_BM = 128;
constexpr int GEMM_BN = 256;
constexpr int GEMM_BK = 128;
constexpr int GEMM_MAX_GROUPS = 1024;
constexpr int GEMM_DENSE_CLUSTER = 2;   // dense GEMM: CTA pairs; each CTA loads half of the W tile

// Device error word codes (the first error of a launch wins).
enum DeviceError : int {
    DEV_OK = 0,
    DEV_TIMEOUT_PRODUCER = 1,   // TMA producer: a smem stage never became free
    DEV_TIMEOUT_MMA_TMEM = 2,   // MMA issuer: a TMEM accumulator buffer never drained
    DEV_TIMEOUT_MMA_FULL = 3,   // MMA issuer: a smem stage never filled
    DEV_TIMEOUT_EPILOGUE = 4,   // epilogue: a K-block partial never arrived
    DEV_TIMEOUT_DRAIN = 5,      // clean-up: in-flight copies or MMAs did not finish
    DEV_TIMEOUT_SCALES = 6,     // scale loader: a scale slot never became free
};

struct GemmArgs {
    const float* a_s;         // [K/128][rows]
    const float* w_s;         // [G][ceil(N/128)][K/128]
    void* c;                  // [rows][ldc]
    int64_t ldc;
    int64_t rows;             // M (dense) or R (grouped)
    int N;
    int KB;                   // K / 128
    int NB;                   // ceil(N / 128)
    int NT;                   // ceil(N / GEMM_BN)
    int MT;                   // dense: ceil(M / 128)
    int num_tiles;            // dense: work items = ceil(MT / cluster) * NT (grouped: on device)
    const int32_t* offsets;   // grouped: [G+1] on the device
    float* h_s;               // output scales, codes go to c: GROUPED_SWIGLU [N/256][rows],
                              // DENSE_QUANT [N/128][rows]
    int G;
    int* err;                 // device error word
    long long budget;         // spin-wait budget in SM clock cycles
    int fault_skip_release;   // test hook: accumulation index at which one epilogue warp skips
                              // its TMEM release (-1: never); set by fp8bs_debug_skip_release
    int band;                 // dense: m-groups per band of the tile order (see gemm_band)
};

// ue8m0: power-of-two tile scales (tile_scale_ue8m0) instead of amax / 448
cudaError_t launch_quant_act(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                             int64_t ldq, float* scales, bool ue8m0, cudaStream_t stream);
cudaError_t launch_quant_weight(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                int64_t ldq, float* scales, bool ue8m0, cudaStream_t stream);
cudaError_t launch_moe_permute(const uint8_t* q, int64_t ldq, const float* s, int64_t T,
                               const int32_t* tok, int64_t R, int64_t K, uint8_t* qp,
                               int64_t ldqp, float* sp, cudaStream_t stream);
cudaError_t launch_moe_combine(const void* y, int64_t ldy, int64_t R, const int32_t* row,
                               const float* w, int64_t T, int64_t topk, int64_t N, void* out,
                               int64_t ldo, cudaStream_t stream);
cudaError_t launch_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* qt,
                                   int64_t ldqt, float* scales, cudaStream_t stream);
cudaError_t launch_quant_weight_t(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* qt,
                                  int64_t ldqt, float* scales_t, cudaStream_t stream);
// max_ctas: the persistent grid's upper bound (the SM count); the launcher sizes the grid.
// One-shot test hook (api.cu): the index for GemmArgs::fault_skip_release of the next grouped
// GEMM launch, then back to -1.
int take_fault_skip_release();

// Few-row GEMM (M <= GEMM_SMALL_MAX_M) computed as C^T = W A^T with split-K over a cluster (gemm_small.cu).
struct SmallArgs {
    const float* a_s;         // [K/128][M]
    const float* w_s;         // [ceil(N/128)][K/128]
    void* c;                  // [M][ldc]
    int64_t ldc;
    int M;
    int N;
    int KB;                   // K / 128
    int n_tiles;              // ceil(N / 128): weight-row tiles
    int m_tiles;              // ceil(M / tokens per tile)
    int split;                // CTAs per cluster sharing one tile's K loop (1, 2, 4 or 8)
    int* err;
    long long budget;
};
constexpr int GEMM_SMALL_MAX_M = 64;   // above this the tiled CTA-pair kernel is faster
int gemm_small_tokens(int64_t M);   // tokens per tile for M rows: 32 or 64
// max_ctas: the persistent grid's upper bound when the K loop is not split (the SM count)
cudaError_t launch_gemm_small(const CUtensorMap& map_w, const CUtensorMap& map_a,
                              const SmallArgs& args, int bnt, bool out_f32, int max_ctas,
                              cudaStream_t stream);

// DENSE: per-128x128-block B scales; GROUPED: the same per expert; ROW_SCALED: a scale per B
// row and K block (the 1d1d weight-gradient GEMM), dense only.
// GROUPED_SWIGLU: grouped, gate/up rows interleaved per 128, epilogue silu(gate) * up re-quantized
// to E4M3 with 1x128 scales.
// DENSE_QUANT: dense, output re-quantized to E4M3 codes with 1x128 scales.
enum class GemmKind { DENSE, GROUPED, ROW_SCALED, GROUPED_SWIGLU, DENSE_QUANT };
// map_c: the output C as BF16 / FP32 with 64-byte boxes of 32 rows (make_out_map); read by the
// kinds whose output is BF16 or FP32 (not GROUPED_SWIGLU or DENSE_QUANT, which take any map).
// store_warp: DENSE with BF16 output or DENSE_QUANT only, the variant whose output tiles are
// written by a store warp while the epilogue goes on (for K loops of 32+ blocks and 4+ tiles per
// pair).
cudaError_t launch_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b,
                        const CUtensorMap& map_c, const GemmArgs& args, GemmKind kind,
                        bool out_f32, int max_ctas, cudaStream_t stream,
                        bool store_warp = false);
int gemm_cluster_size(bool grouped);
// Dense tile order: m-groups (of cluster-size m-tiles) per band for a problem of `mgroups` x `NT`
// items with K bytes of codes per row, on `clusters` concurrent clusters.
int gemm_band(int mgroups, int NT, int64_t K, int clusters);
size_t gemm_smem_bytes(GemmKind kind, int G);

// ------------------------------------------------------------------------------------
// Host-side helpers of the C ABI (api.cu)
// ------------------------------------------------------------------------------------
namespace host {

constexpr int MAX_DEVICES = 64;

struct DeviceInfo {
    int checked = 0;      // 0 unknown, 1 sm_103, -1 other
    int num_sms = 0;
    int* err = nullptr;   // device error word (allocated on first use)
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FP8BS_OK : FP8BS_ERR_CUDA; }

long long wait_budget();
int current_device(DeviceInfo** info);
int ensure_error_word(DeviceInfo* d);
int ensure_encoder();
int make_code_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows, int64_t ld,
                  int box_rows);
// The GEMM output [rows][ld] of BF16 or FP32 as a TMA store target: boxes of 64 bytes x 32 rows
// with the 64-byte swizzle.
int make_out_map(CUtensorMap* map, void* c, int64_t cols, int64_t rows, int64_t ld, bool f32);
int check_quant_args(const void* in, int64_t rows, int64_t K, int64_t ld_in, const void* q,
                     int64_t ldq, const void* scales);
int check_gemm_args(const void* a_q, const void* a_s, const void* w_q, const void* w_s,
                    int64_t rows, int64_t N, int64_t K, const void* c, int64_t ldc, int out_dtype);
// The dense GEMM dispatch after the argument checks (M > 0), with the error word `err`.
int dense_gemm_launch(DeviceInfo* d, int* err, GemmKind kind, const uint8_t* a_q,
                      const float* a_s, const uint8_t* w_q, const float* w_s, int64_t M, int64_t N,
                      int64_t K, void* c, int64_t ldc, int out_dtype, fp8bs_stream_t stream,
                      float* c_s);
// Reads and clears the allocation-free entry point's error word on the current device (if that
// entry point has run there); *timeout is set when a launch recorded a timeout (noalloc.cu).
int noalloc_take_error(bool* timeout);

}  // namespace host

}  // namespace fp8bs
