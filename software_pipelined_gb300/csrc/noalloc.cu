// Split-K GEMM that allocates nothing: gemm_f32_run_splitk_noalloc.
//
// Some callers cannot allocate device memory at the point where they need a
// GEMM: code that runs while a memory pool or allocator is being set up or
// torn down, code under a strict no-allocation budget or arena (the caller owns
// all device memory and hands out only the operands), or a real-time path that
// must not take the allocator's locks or risk its latency.  gemm_f32_plan
// cannot serve them, because a plan allocates its scratch with cudaMalloc.
//
// This entry point runs the SIMT FFMA kernel in split-K mode and keeps the
// per-split partial products in one fixed array that is part of the library
// image (a file-scope __device__ array).  Every GPU that loads the library
// holds that array, 8 MiB of it, until the process exits.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"

namespace gemm_f32 {
namespace {

// 8 MiB of partial sums: (K-slices that run) * M * round_up(N, 4) floats must fit.
constexpr int64_t kNoAllocScratchFloats = int64_t(2) << 20;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

// Device address of the scratch array in the current context.  In host code
// the array's name is only a stand-in, never a device address, so every call
// looks the address up (a table lookup that allocates nothing).  Looking it up
// each time, rather than caching it per device, keeps it right when the
// device's primary context is destroyed and created again in this process
// (the array may then sit at another address).
cudaError_t scratch_for_current_context(float** out)
{
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = static_cast<float*>(p);
    return cudaSuccess;
}

}  // namespace
}  // namespace gemm_f32

using namespace gemm_f32;

extern "C" gemm_f32_status gemm_f32_run_splitk_noalloc(int64_t M, int64_t N, int64_t K, int64_t lda,
                                                       int64_t ldb, int64_t ldc, const float* A,
                                                       const float* B, float* C, int32_t split_k,
                                                       gemm_f32_stream_t stream)
{
    if (M < 0 || N < 0 || K < 0 || lda < 1 || ldb < 1 || ldc < 1) return GEMM_F32_ERR_INVALID_ARG;
    if ((M > 0 && K > 0 && lda < K) || (K > 0 && N > 0 && ldb < N) || (M > 0 && N > 0 && ldc < N))
        return GEMM_F32_ERR_INVALID_ARG;
    if (split_k < 2 || split_k > 64) return GEMM_F32_ERR_INVALID_ARG;
    const int64_t lim = int64_t(1) << 31;
    if (M >= lim || N >= lim || K >= lim) return GEMM_F32_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_F32_OK;
    if (!C || (K > 0 && (!A || !B))) return GEMM_F32_ERR_INVALID_ARG;

    int dev = -1, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_F32_ERR_UNSUPPORTED;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return GEMM_F32_ERR_UNSUPPORTED;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) return zero_fill_launch(C, M, N, ldc, s) == cudaSuccess ? GEMM_F32_OK : GEMM_F32_ERR_CUDA;

    const int cfg = simt_find_config(64, 64, 2);
    if (cfg < 0) return GEMM_F32_ERR_UNSUPPORTED;
    const int64_t bk = simt_config(cfg).bk;
    int64_t chunk = ((K + split_k - 1) / split_k + bk - 1) / bk * bk;
    const int64_t splits = (K + chunk - 1) / chunk;  // no empty K-slice
    const int64_t ldp = (N + 3) / 4 * 4;
    // A single K-slice writes C directly and needs no scratch.  M * ldp < 2^62,
    // so the comparison cannot overflow.
    float* scratch = nullptr;
    if (splits > 1) {
        if (M * ldp > kNoAllocScratchFloats / splits) return GEMM_F32_ERR_INVALID_ARG;
        if (scratch_for_current_context(&scratch) != cudaSuccess) return GEMM_F32_ERR_CUDA;
    }

    SimtArgs a{};
    a.M = M; a.N = N; a.K = K;
    a.A = A; a.lda = lda; a.B = B; a.ldb = ldb; a.C = C; a.ldc = ldc;
    a.split_k = (int)splits;
    a.k_chunk = chunk;
    a.partial = scratch;  // every partial is written in full before it is read
    a.ldp = ldp;
    cudaError_t e = simt_launch(cfg, a, s);
    if (e == cudaSuccess && splits > 1) e = splitk_reduce_launch(scratch, (int)splits, M, N, ldp, C, ldc, s);
    return e == cudaSuccess ? GEMM_F32_OK : GEMM_F32_ERR_CUDA;
}
