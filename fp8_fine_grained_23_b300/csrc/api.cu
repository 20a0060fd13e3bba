// api.cu -- the C ABI declared in include/fp8bs.h: argument checks, device checks, TMA
// descriptors, the per-device error word, and kernel dispatch. Everything is asynchronous on the
// caller's stream; nothing here synchronizes except fp8bs_last_error().
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "fp8bs.h"
#include "internal.h"

using namespace fp8bs;
using namespace fp8bs::host;

namespace fp8bs {
namespace host {

std::mutex g_mu;
int g_fault_skip_release = -1;
DeviceInfo g_dev[MAX_DEVICES];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Default spin-wait budget: 2^31 SM cycles, about one second at the B300's clocks.
long long wait_budget()
{
    static long long budget = [] {
        const char* e = std::getenv("FP8BS_WAIT_BUDGET_CYCLES");
        long long v = e ? std::atoll(e) : 0;
        return v > 0 ? v : (1LL << 31);
    }();
    return budget;
}


// Current device, checked to be compute capability 10.3; fills *info.
int current_device(DeviceInfo** info)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.checked == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        d.checked = (major == 10 && minor == 3) ? 1 : -1;
        d.num_sms = sms;
    }
    if (d.checked != 1) return FP8BS_ERR_UNSUPPORTED_DEVICE;
    *info = &d;
    return FP8BS_OK;
}

int ensure_error_word(DeviceInfo* d)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (d->err) return FP8BS_OK;
    int* p = nullptr;
    if (cudaMalloc(&p, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p);
        return FP8BS_ERR_CUDA;
    }
    d->err = p;
    return FP8BS_OK;
}

int ensure_encoder()
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode) return FP8BS_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return FP8BS_OK;
}

// 2-D map over a row-major byte matrix [rows][cols] (row stride `ld` bytes), loaded in boxes of
// 128 bytes x box_rows rows with the 128-byte swizzle; out-of-range rows read as zero.
int make_code_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows, int64_t ld,
                  int box_rows)
{
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
    const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8BS_OK : FP8BS_ERR_CUDA;
}

int make_out_map(CUtensorMap* map, void* c, int64_t cols, int64_t rows, int64_t ld, bool f32)
{
    const int64_t elem = f32 ? 4 : 2;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * elem)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(64 / elem), 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          2, c, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8BS_OK : FP8BS_ERR_CUDA;
}

int check_quant_args(const void* in, int64_t rows, int64_t K, int64_t ld_in, const void* q,
                     int64_t ldq, const void* scales)
{
    if (rows < 0 || K <= 0 || K % 128 != 0 || ld_in < K || ldq < K) return FP8BS_ERR_INVALID_ARG;
    if (rows > INT32_MAX || K > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (rows == 0) return FP8BS_OK;
    if (!in || !q || !scales) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(in) || !aligned16(q) || !aligned4(scales) || ld_in % 8 != 0 || ldq % 16 != 0)
        return FP8BS_ERR_MISALIGNED;
    return FP8BS_OK;
}

int check_gemm_args(const void* a_q, const void* a_s, const void* w_q, const void* w_s,
                    int64_t rows, int64_t N, int64_t K, const void* c, int64_t ldc, int out_dtype)
{
    if (out_dtype != FP8BS_OUT_BF16 && out_dtype != FP8BS_OUT_F32) return FP8BS_ERR_INVALID_ARG;
    if (rows < 0 || N <= 0 || N % 16 != 0 || K <= 0 || K % 128 != 0 || ldc < N)
        return FP8BS_ERR_INVALID_ARG;
    if (rows > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (rows == 0) return FP8BS_OK;
    if (!a_q || !a_s || !w_q || !w_s || !c) return FP8BS_ERR_INVALID_ARG;
    const int64_t elem = out_dtype == FP8BS_OUT_F32 ? 4 : 2;
    if (!aligned16(a_q) || !aligned16(w_q) || !aligned16(c) || !aligned4(a_s) || !aligned4(w_s) ||
        (ldc * elem) % 16 != 0)
        return FP8BS_ERR_MISALIGNED;
    return FP8BS_OK;
}

// Transposing quantizers: the rows are the contracted index of the later GEMM, in blocks of
// 128 (rows % 128 == 0); codes [K][ldqt >= rows].
int check_transpose_quant_args(const void* in, int64_t rows, int64_t K, int64_t ld_in,
                               const void* qt, int64_t ldqt, const void* scales)
{
    if (rows < 0 || rows % 128 != 0 || K <= 0 || K % 128 != 0 || ld_in < K || ldqt < rows)
        return FP8BS_ERR_INVALID_ARG;
    if (rows > INT32_MAX || K > INT32_MAX || rows / 128 > 65535) return FP8BS_ERR_INVALID_ARG;
    if (rows == 0) return FP8BS_OK;
    if (!in || !qt || !scales) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(in) || !aligned16(qt) || !aligned4(scales) || ld_in % 8 != 0 ||
        ldqt % 16 != 0)
        return FP8BS_ERR_MISALIGNED;
    return FP8BS_OK;
}

// Dense GEMM launch shared by fp8_blockscaled_gemm (block-scaled W), fp8_blockscaled_gemm_1d1d
// (per-row B scales), fp8_blockscaled_gemm_quant and the allocation-free entry point: the same
// dispatch (few-row kernel for M <= GEMM_SMALL_MAX_M, else the CTA-pair kernel), tiles, maps and
// persistent grid. The arguments have been checked and M > 0; `err` is the device error word the
// kernels record a timeout in.
int dense_gemm_launch(DeviceInfo* d, int* err, GemmKind kind, const uint8_t* a_q,
                      const float* a_s, const uint8_t* w_q, const float* w_s, int64_t M, int64_t N,
                      int64_t K, void* c, int64_t ldc, int out_dtype, fp8bs_stream_t stream,
                      float* c_s)
{
    int st = FP8BS_OK;
    if ((st = ensure_encoder()) != FP8BS_OK) return st;

    if (kind == GemmKind::DENSE && M <= GEMM_SMALL_MAX_M) {
        // Few rows: the weight rows take the tensor core's 128-row side, the M rows its narrow
        // side; the K loop is split over a cluster while the weight tiles cannot cover the SMs.
        const int bnt = gemm_small_tokens(M);
        CUtensorMap mw, ma;
        if ((st = make_code_map(&mw, w_q, K, N, K, 128)) != FP8BS_OK) return st;
        if ((st = make_code_map(&ma, a_q, K, M, K, bnt)) != FP8BS_OK) return st;
        SmallArgs sa{};
        sa.a_s = a_s;
        sa.w_s = w_s;
        sa.c = c;
        sa.ldc = ldc;
        sa.M = static_cast<int>(M);
        sa.N = static_cast<int>(N);
        sa.KB = static_cast<int>(K / 128);
        sa.n_tiles = static_cast<int>((N + 127) / 128);
        sa.m_tiles = static_cast<int>((M + bnt - 1) / bnt);
        sa.split = 1;
        const int64_t items = static_cast<int64_t>(sa.n_tiles) * sa.m_tiles;
        while (sa.split < 8 && items * sa.split * 2 <= d->num_sms && sa.KB >= 4 * sa.split)
            sa.split *= 2;
        if (items * sa.split > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
        sa.err = err;
        sa.budget = wait_budget();
        return cuda_status(launch_gemm_small(mw, ma, sa, bnt, out_dtype == FP8BS_OUT_F32,
                                             d->num_sms, reinterpret_cast<cudaStream_t>(stream)));
    }

    const int cluster = gemm_cluster_size(false);
    CUtensorMap ma, mb, mc;
    if ((st = make_code_map(&ma, a_q, K, M, K, GEMM_BM)) != FP8BS_OK) return st;
    if ((st = make_code_map(&mb, w_q, K, N, K, GEMM_BN / cluster)) != FP8BS_OK) return st;
    if (kind == GemmKind::DENSE_QUANT)
        mc = ma;   // (the re-quantized output stores its codes itself)
    else if ((st = make_out_map(&mc, c, N, M, ldc, out_dtype == FP8BS_OUT_F32)) != FP8BS_OK)
        return st;

    GemmArgs args{};
    args.a_s = a_s;
    args.w_s = w_s;
    args.c = c;
    args.ldc = ldc;
    args.rows = M;
    args.N = static_cast<int>(N);
    args.KB = static_cast<int>(K / 128);
    args.NB = static_cast<int>((N + 127) / 128);
    args.NT = static_cast<int>((N + GEMM_BN - 1) / GEMM_BN);
    args.MT = static_cast<int>((M + GEMM_BM - 1) / GEMM_BM);
    const int64_t items = static_cast<int64_t>((args.MT + cluster - 1) / cluster) * args.NT;
    if (items > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    args.num_tiles = static_cast<int>(items);
    args.band = gemm_band((args.MT + cluster - 1) / cluster, args.NT, K, d->num_sms / cluster);
    // the store warp: BF16 dense output or re-quantized codes, K loops of at least 32 blocks,
    // 4+ tiles per pair
    const bool store_warp =
        ((kind == GemmKind::DENSE && out_dtype == FP8BS_OUT_BF16) || kind == GemmKind::DENSE_QUANT) &&
        args.KB >= 32 && items >= 4 * static_cast<int64_t>(d->num_sms / cluster);
    args.offsets = nullptr;
    args.h_s = c_s;
    args.G = 1;
    args.err = err;
    args.budget = wait_budget();
    args.fault_skip_release = -1;
    return cuda_status(launch_gemm(ma, mb, mc, args, kind, out_dtype == FP8BS_OUT_F32, d->num_sms,
                                   reinterpret_cast<cudaStream_t>(stream), store_warp));
}

int dense_gemm(GemmKind kind, const uint8_t* a_q, const float* a_s, const uint8_t* w_q,
               const float* w_s, int64_t M, int64_t N, int64_t K, void* c, int64_t ldc,
               int out_dtype, fp8bs_stream_t stream, float* c_s = nullptr)
{
    int st = kind == GemmKind::DENSE_QUANT ? FP8BS_OK
                                           : check_gemm_args(a_q, a_s, w_q, w_s, M, N, K, c, ldc,
                                                             out_dtype);
    if (st != FP8BS_OK || M == 0) return st;
    DeviceInfo* d = nullptr;
    if ((st = current_device(&d)) != FP8BS_OK) return st;
    if ((st = ensure_error_word(d)) != FP8BS_OK) return st;
    return dense_gemm_launch(d, d->err, kind, a_q, a_s, w_q, w_s, M, N, K, c, ldc, out_dtype,
                             stream, c_s);
}

// Grouped launch shared by the plain grouped GEMM and the SwiGLU + re-quantizing one; the
// caller has checked the output arguments (and that R > 0).
int grouped_gemm(GemmKind kind, const uint8_t* a_q, const float* a_s, const uint8_t* w_q,
                 const float* w_s, const int32_t* group_offsets, int64_t G, int64_t R, int64_t N,
                 int64_t K, void* c, int64_t ldc, bool out_f32, float* h_s,
                 fp8bs_stream_t stream)
{
    int st = FP8BS_OK;
    if (!group_offsets) return FP8BS_ERR_INVALID_ARG;
    if (!aligned4(group_offsets)) return FP8BS_ERR_MISALIGNED;
    if (G * N > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    if ((st = current_device(&d)) != FP8BS_OK) return st;
    if ((st = ensure_error_word(d)) != FP8BS_OK) return st;
    if ((st = ensure_encoder()) != FP8BS_OK) return st;

    CUtensorMap ma, mb, mc;
    if ((st = make_code_map(&ma, a_q, K, R, K, GEMM_BM)) != FP8BS_OK) return st;
    if ((st = make_code_map(&mb, w_q, K, G * N, K, GEMM_BN)) != FP8BS_OK) return st;
    if (kind == GemmKind::GROUPED_SWIGLU)
        mc = ma;   // (the fused epilogue stores its codes itself)
    else if ((st = make_out_map(&mc, c, N, R, ldc, out_f32)) != FP8BS_OK)
        return st;

    GemmArgs args{};
    args.a_s = a_s;
    args.w_s = w_s;
    args.c = c;
    args.ldc = ldc;
    args.rows = R;
    args.N = static_cast<int>(N);
    args.KB = static_cast<int>(K / 128);
    args.NB = static_cast<int>((N + 127) / 128);
    args.NT = static_cast<int>((N + GEMM_BN - 1) / GEMM_BN);
    args.MT = 0;
    args.num_tiles = 0;
    args.band = 1;
    args.offsets = group_offsets;
    args.h_s = h_s;
    args.G = static_cast<int>(G);
    args.err = d->err;
    args.budget = wait_budget();
    args.fault_skip_release = take_fault_skip_release();
    // At most ceil(R/128) + G m-tiles exist across the groups; the exact count is formed on the
    // device from the offsets, and CTAs without a tile exit at once.
    const int64_t bound = ((R + GEMM_BM - 1) / GEMM_BM + G) * args.NT;
    if (bound > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    const int max_ctas = static_cast<int>(bound < d->num_sms ? bound : d->num_sms);
    return cuda_status(
        launch_gemm(ma, mb, mc, args, kind, out_f32, max_ctas, reinterpret_cast<cudaStream_t>(stream)));
}

// The two tile quantizers, with amax/448 or power-of-two (ue8m0) scales.
int quant_act(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
              float* scales, bool ue8m0, fp8bs_stream_t stream)
{
    int st = check_quant_args(x, M, K, ldx, q, ldq, scales);
    if (st != FP8BS_OK || M == 0) return st;
    DeviceInfo* d = nullptr;
    if ((st = current_device(&d)) != FP8BS_OK) return st;
    return cuda_status(launch_quant_act(x, M, K, ldx, q, ldq, scales, ue8m0,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int quant_weight(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, int64_t ldq,
                 float* scales, bool ue8m0, fp8bs_stream_t stream)
{
    int st = check_quant_args(w, N, K, ldw, q, ldq, scales);
    if (st != FP8BS_OK || N == 0) return st;
    if ((N + 127) / 128 > 65535) return FP8BS_ERR_INVALID_ARG;   // grid.y limit
    DeviceInfo* d = nullptr;
    if ((st = current_device(&d)) != FP8BS_OK) return st;
    return cuda_status(launch_quant_weight(w, N, K, ldw, q, ldq, scales, ue8m0,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace host

int take_fault_skip_release()
{
    std::lock_guard<std::mutex> lock(host::g_mu);
    const int v = host::g_fault_skip_release;
    host::g_fault_skip_release = -1;
    return v;
}

}  // namespace fp8bs

extern "C" {

int fp8_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                        float* scales, fp8bs_stream_t stream)
{
    return fp8bs::host::quant_act(x, M, K, ldx, q, ldq, scales, false, stream);
}

int fp8_quant_act_1x128_ue8m0(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                              int64_t ldq, float* scales, fp8bs_stream_t stream)
{
    return fp8bs::host::quant_act(x, M, K, ldx, q, ldq, scales, true, stream);
}

int fp8_quant_weight_128x128(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                             int64_t ldq, float* scales, fp8bs_stream_t stream)
{
    return fp8bs::host::quant_weight(w, N, K, ldw, q, ldq, scales, false, stream);
}

int fp8_quant_weight_128x128_ue8m0(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                   int64_t ldq, float* scales, fp8bs_stream_t stream)
{
    return fp8bs::host::quant_weight(w, N, K, ldw, q, ldq, scales, true, stream);
}

int fp8_blockscaled_gemm(const uint8_t* a_q, const float* a_s, const uint8_t* w_q,
                         const float* w_s, int64_t M, int64_t N, int64_t K, void* c, int64_t ldc,
                         int out_dtype, fp8bs_stream_t stream)
{
    return fp8bs::host::dense_gemm(GemmKind::DENSE, a_q, a_s, w_q, w_s, M, N, K, c, ldc,
                                   out_dtype, stream);
}

int fp8_blockscaled_gemm_1d1d(const uint8_t* a_q, const float* a_s, const uint8_t* b_q,
                              const float* b_s, int64_t M, int64_t N, int64_t K, void* c,
                              int64_t ldc, int out_dtype, fp8bs_stream_t stream)
{
    return fp8bs::host::dense_gemm(GemmKind::ROW_SCALED, a_q, a_s, b_q, b_s, M, N, K, c, ldc,
                                   out_dtype, stream);
}

int fp8_blockscaled_gemm_quant(const uint8_t* a_q, const float* a_s, const uint8_t* w_q,
                               const float* w_s, int64_t M, int64_t N, int64_t K, uint8_t* c_q,
                               int64_t ldcq, float* c_s, fp8bs_stream_t stream)
{
    if (M < 0 || N <= 0 || N % 128 != 0 || K <= 0 || K % 128 != 0 || ldcq < N)
        return FP8BS_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (M == 0) return FP8BS_OK;
    if (!a_q || !a_s || !w_q || !w_s || !c_q || !c_s) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(a_q) || !aligned16(w_q) || !aligned16(c_q) || !aligned4(a_s) ||
        !aligned4(w_s) || !aligned4(c_s) || ldcq % 16 != 0)
        return FP8BS_ERR_MISALIGNED;
    return fp8bs::host::dense_gemm(GemmKind::DENSE_QUANT, a_q, a_s, w_q, w_s, M, N, K, c_q, ldcq,
                                   FP8BS_OUT_BF16, stream, c_s);
}

int fp8_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* qt,
                        int64_t ldqt, float* scales, fp8bs_stream_t stream)
{
    int st = check_transpose_quant_args(x, M, K, ldx, qt, ldqt, scales);
    if (st != FP8BS_OK || M == 0) return st;
    DeviceInfo* d = nullptr;
    if ((st = current_device(&d)) != FP8BS_OK) return st;
    return cuda_status(launch_quant_act_128x1(x, M, K, ldx, qt, ldqt, scales,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

int fp8_quant_weight_128x128_t(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* qt,
                               int64_t ldqt, float* scales_t, fp8bs_stream_t stream)
{
    int st = check_transpose_quant_args(w, N, K, ldw, qt, ldqt, scales_t);
    if (st != FP8BS_OK || N == 0) return st;
    DeviceInfo* d = nullptr;
    if ((st = current_device(&d)) != FP8BS_OK) return st;
    return cuda_status(launch_quant_weight_t(w, N, K, ldw, qt, ldqt, scales_t,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int fp8_blockscaled_grouped_gemm(const uint8_t* a_q, const float* a_s, const uint8_t* w_q,
                                 const float* w_s, const int32_t* group_offsets, int64_t G,
                                 int64_t R, int64_t N, int64_t K, void* c, int64_t ldc,
                                 int out_dtype, fp8bs_stream_t stream)
{
    if (G < 1 || G > GEMM_MAX_GROUPS) return FP8BS_ERR_INVALID_ARG;
    int st = check_gemm_args(a_q, a_s, w_q, w_s, R, N, K, c, ldc, out_dtype);
    if (st != FP8BS_OK || R == 0) return st;
    return fp8bs::host::grouped_gemm(GemmKind::GROUPED, a_q, a_s, w_q, w_s, group_offsets, G, R,
                                     N, K, c, ldc, out_dtype == FP8BS_OUT_F32, nullptr, stream);
}

int fp8_blockscaled_grouped_gemm_swiglu_quant(const uint8_t* a_q, const float* a_s,
                                              const uint8_t* w_q, const float* w_s,
                                              const int32_t* group_offsets, int64_t G, int64_t R,
                                              int64_t N2, int64_t K, uint8_t* h_q, int64_t ldh,
                                              float* h_s, fp8bs_stream_t stream)
{
    if (G < 1 || G > GEMM_MAX_GROUPS) return FP8BS_ERR_INVALID_ARG;
    if (R < 0 || N2 <= 0 || N2 % 256 != 0 || K <= 0 || K % 128 != 0 || ldh < N2 / 2)
        return FP8BS_ERR_INVALID_ARG;
    if (R > INT32_MAX || N2 > INT32_MAX || K > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (R == 0) return FP8BS_OK;
    if (!a_q || !a_s || !w_q || !w_s || !h_q || !h_s) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(a_q) || !aligned16(w_q) || !aligned16(h_q) || !aligned4(a_s) ||
        !aligned4(w_s) || !aligned4(h_s) || ldh % 16 != 0)
        return FP8BS_ERR_MISALIGNED;
    return fp8bs::host::grouped_gemm(GemmKind::GROUPED_SWIGLU, a_q, a_s, w_q, w_s, group_offsets,
                                     G, R, N2, K, h_q, ldh, false, h_s, stream);
}

int fp8_moe_permute(const uint8_t* q, int64_t ldq, const float* s, int64_t T,
                    const int32_t* token_of_row, int64_t R, int64_t K, uint8_t* qp, int64_t ldqp,
                    float* sp, fp8bs_stream_t stream)
{
    if (T < 0 || R < 0 || K <= 0 || K % 128 != 0 || ldq < K || ldqp < K) return FP8BS_ERR_INVALID_ARG;
    if (T > INT32_MAX || R > INT32_MAX || K > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (R == 0) return FP8BS_OK;
    if (T == 0 || !q || !s || !token_of_row || !qp || !sp) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(qp) || ldq % 16 != 0 || ldqp % 16 != 0 || !aligned4(s) ||
        !aligned4(sp) || !aligned4(token_of_row))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    int st = current_device(&d);
    if (st != FP8BS_OK) return st;
    return cuda_status(launch_moe_permute(q, ldq, s, T, token_of_row, R, K, qp, ldqp, sp,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int fp8_moe_combine(const void* y, int64_t ldy, int64_t R, const int32_t* row_of_token,
                    const float* weights, int64_t T, int64_t topk, int64_t N, void* out,
                    int64_t ldo, fp8bs_stream_t stream)
{
    if (R < 0 || T < 0 || topk < 1 || topk > 32 || N <= 0 || N % 8 != 0 || ldy < N || ldo < N)
        return FP8BS_ERR_INVALID_ARG;
    if (R > INT32_MAX || T > INT32_MAX || N > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (T == 0) return FP8BS_OK;
    if (!y || !row_of_token || !weights || !out) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(out) || ldy % 8 != 0 || ldo % 8 != 0 ||
        !aligned4(row_of_token) || !aligned4(weights))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    int st = current_device(&d);
    if (st != FP8BS_OK) return st;
    return cuda_status(launch_moe_combine(y, ldy, R, row_of_token, weights, T, topk, N, out, ldo,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int fp8bs_debug_skip_release(int at)
{
    if (at < 0) return FP8BS_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    g_fault_skip_release = at;
    return FP8BS_OK;
}

const char* fp8bs_status_string(int status)
{
    switch (status) {
        case FP8BS_OK: return "FP8BS_OK";
        case FP8BS_ERR_INVALID_ARG: return "FP8BS_ERR_INVALID_ARG";
        case FP8BS_ERR_MISALIGNED: return "FP8BS_ERR_MISALIGNED";
        case FP8BS_ERR_UNSUPPORTED_DEVICE: return "FP8BS_ERR_UNSUPPORTED_DEVICE";
        case FP8BS_ERR_CUDA: return "FP8BS_ERR_CUDA";
        case FP8BS_ERR_TIMEOUT: return "FP8BS_ERR_TIMEOUT";
        default: return "FP8BS_ERR_UNKNOWN";
    }
}

int fp8bs_last_error(fp8bs_stream_t stream)
{
    DeviceInfo* d = nullptr;
    int st = current_device(&d);
    if (st != FP8BS_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    // The allocation-free GEMM records its timeouts in its own word inside the library image.
    bool noalloc_timeout = false;
    if ((st = noalloc_take_error(&noalloc_timeout)) != FP8BS_OK) return st;
    if (!d->err) return noalloc_timeout ? FP8BS_ERR_TIMEOUT : FP8BS_OK;
    int h = 0;
    if (cudaMemcpy(&h, d->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    if (h == DEV_OK) return noalloc_timeout ? FP8BS_ERR_TIMEOUT : FP8BS_OK;
    if (cudaMemset(d->err, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    return FP8BS_ERR_TIMEOUT;
}

}  // extern "C"
