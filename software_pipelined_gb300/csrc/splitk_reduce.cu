// Deterministic split-K reduction and the K == 0 zero fill.
//
// With split-K each K-slice's kernel writes its partial product to scratch,
// P[z] (z = 0 .. splits-1, each M x ldp).  This kernel forms
// C[i][j] = P[0][i][j] + P[1][i][j] + ... in ascending z, always in the same
// order, so repeated runs give bit-identical C.  HBM-bound: it reads
// splits*M*N and writes M*N floats, 16 bytes per access where the rows allow,
// with a grid-stride loop over a grid sized to the SM count.
#include <cstdint>

#include "internal.h"

namespace gemm_f32 {
namespace {

// Programmatic serialisation: this kernel may be launched while the split-K
// GEMM before it finishes, and waits for it before reading its partials.  It
// releases its own successor only by completing: a successor's CTAs waiting
// early would take the slots these blocks need.
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

__global__ void __launch_bounds__(256)
splitk_reduce_vec4(const float4* __restrict__ P, int splits, int64_t M, int64_t n4,
                   int64_t ldp4, int64_t slice4, float4* __restrict__ C, int64_t ldc4)
{
    pdl_enter();
    const int64_t total = M * n4;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / n4, j = idx % n4;
        const float4* p = P + i * ldp4 + j;
        float4 s = __ldg(p);
        for (int z = 1; z < splits; ++z) {
            const float4 t = __ldg(p + z * slice4);
            s.x += t.x; s.y += t.y; s.z += t.z; s.w += t.w;
        }
        C[i * ldc4 + j] = s;
    }
}

__global__ void __launch_bounds__(256)
splitk_reduce_scalar(const float* __restrict__ P, int splits, int64_t M, int64_t N,
                     int64_t ldp, int64_t slice, float* __restrict__ C, int64_t ldc)
{
    pdl_enter();
    const int64_t total = M * N;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / N, j = idx % N;
        const float* p = P + i * ldp + j;
        float s = __ldg(p);
        for (int z = 1; z < splits; ++z) s += __ldg(p + z * slice);
        C[i * ldc + j] = s;
    }
}

__global__ void __launch_bounds__(256)
zero_fill_kernel(float* __restrict__ C, int64_t M, int64_t N, int64_t ldc)
{
    const int64_t total = M * N;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x)
        C[(idx / N) * ldc + idx % N] = 0.f;
}

int grid_for(int64_t work)
{
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 152;
    }
    const int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;  // 8 resident 256-thread blocks per SM
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t splitk_reduce_launch(const float* P, int splits, int64_t M, int64_t N, int64_t ldp,
                                 float* C, int64_t ldc, cudaStream_t s)
{
    if (M <= 0 || N <= 0) return cudaSuccess;
    const int64_t slice = M * ldp;
    const bool vec = (N % 4 == 0) && (ldp % 4 == 0) && (ldc % 4 == 0) &&
                     (reinterpret_cast<uintptr_t>(C) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(P) % 16 == 0);
    if (vec) {
        const int64_t n4 = N / 4;
        return launch_pdl(splitk_reduce_vec4, grid_for(M * n4), s, reinterpret_cast<const float4*>(P), splits,
                          M, n4, ldp / 4, slice / 4, reinterpret_cast<float4*>(C), ldc / 4);
    }
    return launch_pdl(splitk_reduce_scalar, grid_for(M * N), s, P, splits, M, N, ldp, slice, C, ldc);
}

cudaError_t zero_fill_launch(float* C, int64_t M, int64_t N, int64_t ldc, cudaStream_t s)
{
    if (M <= 0 || N <= 0) return cudaSuccess;
    zero_fill_kernel<<<grid_for(M * N), 256, 0, s>>>(C, M, N, ldc);
    return cudaGetLastError();
}

}  // namespace gemm_f32
