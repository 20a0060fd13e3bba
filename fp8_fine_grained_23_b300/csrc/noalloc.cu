// noalloc.cu -- fp8_blockscaled_gemm_noalloc: the dense block-scaled GEMM for callers that may not
// allocate device memory.
//
// The GEMM kernels need one word of global scratch: the error word in which a CTA records a
// pipeline wait that ran past its budget. fp8_blockscaled_gemm obtains that word with cudaMalloc on
// its first call on a device. Some callers cannot let a library allocate: frameworks that hand
// out all device memory through their own caching allocator or pool and treat any other cudaMalloc
// as an error (it would fragment or overrun the pool's budget), and deployments that must know
// their full device footprint before they start. This entry point runs the same dispatch and
// kernels (the few-row kernel for M <= 64, the CTA-pair kernel above) with their scratch in a fixed
// array that lives in the library image itself (a static __device__ array, loaded on every GPU
// that loads the library and kept until the process exits). Nothing is allocated per call or on
// the first call.
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
constexpr int NOALLOC_WORDS_PER_CALL = 1;   // the kernels' error word

// Zero when the library is loaded. A kernel only ever moves the error word from zero to a
// timeout code (atomic compare-and-swap), and fp8bs_last_error() reads it and puts it back to
// zero, so it needs no clearing per call: a timeout stays recorded until it is read.
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

namespace fp8bs {
namespace host {

int noalloc_take_error(bool* timeout)
{
    *timeout = false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    int* word = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        word = g_noalloc_ptr[dev];
    }
    if (word == nullptr) return FP8BS_OK;   // the entry point never ran on this device
    int h = 0;
    if (cudaMemcpy(&h, word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    if (h == DEV_OK) return FP8BS_OK;
    if (cudaMemset(word, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    *timeout = true;
    return FP8BS_OK;
}

}  // namespace host
}  // namespace fp8bs

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
    return dense_gemm_launch(d, scratch, GemmKind::DENSE, a_q, a_s, w_q, w_s, M, N, K, c, ldc,
                             out_dtype, stream, nullptr);
}
