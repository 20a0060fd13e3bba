// noalloc.cu -- fp8_blockscaled_gemm_noalloc: the dense block-scaled GEMM for callers that may not
// allocate device memory.
//
// The GEMM kernel needs one word of global scratch: the error word in which a CTA records a
// pipeline wait that ran past its budget. fp8_blockscaled_gemm obtains that word with cudaMalloc on
// its first call on a device. Some callers cannot let a library allocate: frameworks that hand
// out all device memory through their own caching allocator or pool and treat any other cudaMalloc
// as an error (it would fragment or overrun the pool's budget), and deployments that must know
// their full device footprint before they start. This entry point runs the same kernel
// with its scratch in a fixed array that lives in the library image itself (a static __device__
// array, loaded on every GPU that loads the library and kept until the process exits). Nothing is
// allocated per call or on the first call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fp8bs.h"
#include "internal.h"

using namespace fp8bs;
using namespace fp8bs::host;

namespace {

// Scratch capacity in 32-bit words (256 bytes). A call needs NOALLOC_WORDS_PER_CALL of them.
constexpr int NOALLOC_SCRATCH_WORDS = 64;
constexpr int NOALLOC_WORDS_PER_CALL = 1;   // the kernel's error word

static __device__ __align__(256) int g_noalloc_scratch[NOALLOC_SCRATCH_WORDS];

std::mutex g_noalloc_mu;
int* g_noalloc_ptr[MAX_DEVICES] = {};

// Device address of the scratch array on the current device `dev`. In host code the name
// g_noalloc_scratch is only a host-side stand-in, so the address is looked up once per device,
// with that device current, and cached.
int noalloc_scratch(int dev, int** out)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = static_cast<int*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return FP8BS_OK;
}

}  // namespace

extern "C" int fp8_blockscaled_gemm_noalloc(const uint8_t* a_q, const float* a_s,
                                            const uint8_t* w_q, const float* w_s, int64_t M,
                                            int64_t N, int64_t K, void* c, int64_t ldc,
                                            int out_dtype, fp8bs_stream_t stream)
{
    int st = check_gemm_args(a_q, a_s, w_q, w_s, M, N, K, c, ldc, out_dtype);
    if (st != FP8BS_OK || M == 0) return st;
    if (NOALLOC_WORDS_PER_CALL > NOALLOC_SCRATCH_WORDS) return FP8BS_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    if ((st = current_device(&d)) != FP8BS_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    int* scratch = nullptr;
    if ((st = noalloc_scratch(dev, &scratch)) != FP8BS_OK) return st;
    if ((st = ensure_encoder()) != FP8BS_OK) return st;

    const int cluster = gemm_cluster_size(false);
    CUtensorMap ma, mb;
    if ((st = make_code_map(&ma, a_q, K, M, K, GEMM_BM)) != FP8BS_OK) return st;
    if ((st = make_code_map(&mb, w_q, K, N, K, GEMM_BN / cluster)) != FP8BS_OK) return st;

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
    args.offsets = nullptr;
    args.G = 1;
    args.err = scratch;   // the error word must start at zero on every call
    args.budget = wait_budget();
    args.fault_skip_release = -1;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, NOALLOC_WORDS_PER_CALL * sizeof(int), s) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    return cuda_status(launch_gemm(ma, mb, args, GemmKind::DENSE, out_dtype == FP8BS_OUT_F32, d->num_sms, s));
}
