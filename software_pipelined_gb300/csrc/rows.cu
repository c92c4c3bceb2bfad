// Products with a short A (M up to 16 rows) against a large B: C = A*B is then
// bound by reading B from HBM once, and tiles of 128 (tensor cores) or 32
// (SIMT) rows would compute mostly padding.  This kernel streams B instead,
// with plain FP32 FMAs (the same accumulation as the SIMT kernel: FP32 sums of
// FP32 products, within the library's bound).
//
// A block takes kRowsCols = 256 columns of B (64 float4) and one K-range (a
// multiple of kRowsK = 256 rows, taken 256 rows at a time).  Its 256 threads
// are 64 column quads x 4 row groups: a thread keeps MR x 4 sums (the rows of
// A, columns n..n+3) over the k of its group (g, g + 4, ... of the range, in
// order), with A's 256-row piece staged in shared memory and read as
// broadcasts.  The 4 groups are added in group order through shared memory,
// and the block writes its K-range's MR x 256 partial (summed in range order
// by the split-K reduction) or, when one range covers K, C itself.  So every
// output is summed in one fixed order, run after run.
#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"

namespace gemm_f32 {
namespace {

constexpr int kRowsCols = 256;
constexpr int kRowsK = 256;
constexpr int kRowsThreads = 256;
constexpr int kRowsGroups = kRowsThreads / (kRowsCols / 4);  // row groups
constexpr int kRowsUnroll = 4;                                // B loads in flight per thread

template <int MR>
__global__ void __launch_bounds__(kRowsThreads)
rows_kernel(const float* __restrict__ A, int64_t lda, const float* __restrict__ B, int64_t ldb,
            float* __restrict__ out, int64_t ldo, int64_t slice, int64_t M, int64_t N, int64_t K, int64_t range,
            int vec_b)
{
    // A's piece during the loop, then the group sums (the larger of the two)
    constexpr int kRed = (kRowsGroups - 1) * MR * kRowsCols;
    constexpr int kWords = kRed > MR * kRowsK ? kRed : MR * kRowsK;
    __shared__ float sm[kWords];
    const int t = threadIdx.x, q = t % (kRowsCols / 4), grp = t / (kRowsCols / 4);
    const int64_t n = (int64_t)blockIdx.x * kRowsCols + 4 * q;
    const int64_t kr0 = (int64_t)blockIdx.y * range;
    const int64_t kr1 = K - kr0 < range ? K : kr0 + range;
    float acc[MR][4];
#pragma unroll
    for (int i = 0; i < MR; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
    const bool quad = vec_b && n + 3 < N;
    for (int64_t k0 = kr0; k0 < kr1; k0 += kRowsK) {
        const int kn = (int)(kr1 - k0 < kRowsK ? kr1 - k0 : kRowsK);
        __syncthreads();  // the previous piece of A is read
        for (int e = t; e < MR * kRowsK; e += kRowsThreads) {
            const int i = e / kRowsK, kk = e % kRowsK;
            sm[e] = (i < M && kk < kn) ? __ldg(A + i * lda + k0 + kk) : 0.f;
        }
        __syncthreads();
        for (int kk = grp; kk < kn; kk += kRowsGroups * kRowsUnroll) {
            float b[kRowsUnroll][4];
#pragma unroll
            for (int u = 0; u < kRowsUnroll; ++u) {
                const int k = kk + u * kRowsGroups;
                const float* row = B + (k0 + k) * ldb + n;
                if (k >= kn) {
                    b[u][0] = b[u][1] = b[u][2] = b[u][3] = 0.f;
                } else if (quad) {
                    const float4 v = __ldg(reinterpret_cast<const float4*>(row));
                    b[u][0] = v.x; b[u][1] = v.y; b[u][2] = v.z; b[u][3] = v.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) b[u][c] = n + c < N ? __ldg(row + c) : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kRowsUnroll; ++u) {
                const int k = kk + u * kRowsGroups;
                if (k < kn) {
#pragma unroll
                    for (int i = 0; i < MR; ++i) {
                        const float a = sm[i * kRowsK + k];
#pragma unroll
                        for (int c = 0; c < 4; ++c) acc[i][c] = fmaf(a, b[u][c], acc[i][c]);
                    }
                }
            }
        }
    }
    __syncthreads();  // A's last piece is read: the buffer takes the group sums
    if (grp > 0) {
#pragma unroll
        for (int i = 0; i < MR; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) sm[((grp - 1) * MR + i) * kRowsCols + 4 * q + c] = acc[i][c];
    }
    __syncthreads();
    if (grp == 0) {
        float* o = out + (int64_t)blockIdx.y * slice;
#pragma unroll
        for (int i = 0; i < MR; ++i) {
            if (i >= M) break;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float v = acc[i][c];
                for (int g = 0; g < kRowsGroups - 1; ++g) v += sm[(g * MR + i) * kRowsCols + 4 * q + c];
                if (n + c < N) o[i * ldo + n + c] = v;
            }
        }
    }
}

template <int MR>
cudaError_t launch_rows(const RowsArgs& a, cudaStream_t s)
{
    const int64_t gx = (a.N + kRowsCols - 1) / kRowsCols, gy = (a.K + a.range - 1) / a.range;
    const bool split = gy > 1;
    const int vec_b = (a.ldb % 4 == 0) && (reinterpret_cast<uintptr_t>(a.B) % 16 == 0);
    rows_kernel<MR><<<dim3((unsigned)gx, (unsigned)gy), kRowsThreads, 0, s>>>(
        a.A, a.lda, a.B, a.ldb, split ? a.partial : a.C, split ? a.ldp : a.ldc, split ? a.M * a.ldp : 0, a.M, a.N,
        a.K, a.range, vec_b);
    return cudaGetLastError();
}

}  // namespace

int64_t rows_range(int64_t N, int64_t K, int sms)
{
    // K-ranges for about 16 blocks per SM in all (a few waves: 2 to 8 fit at
    // once, by the rows' registers), each a whole number of 256-row pieces; the
    // partials then stay under 16 x 256 x 4 bytes a block
    const int64_t gx = (N + kRowsCols - 1) / kRowsCols, pieces = (K + kRowsK - 1) / kRowsK;
    int64_t want = (int64_t)sms * 16 / (gx > 0 ? gx : 1);
    if (want < 1) want = 1;
    if (want > pieces) want = pieces;
    if (want > 65535) want = 65535;
    return (pieces + want - 1) / want * kRowsK;
}

cudaError_t rows_launch(const RowsArgs& a, cudaStream_t s)
{
    if (a.M < 1 || a.M > kRowsMaxM || a.N < 1 || a.K < 1 || a.range < kRowsK || a.range % kRowsK != 0)
        return cudaErrorInvalidValue;
    if ((a.N + kRowsCols - 1) / kRowsCols > 2147483647 || (a.K + a.range - 1) / a.range > 65535)
        return cudaErrorInvalidValue;
    if (a.M <= 1) return launch_rows<1>(a, s);
    if (a.M <= 2) return launch_rows<2>(a, s);
    if (a.M <= 4) return launch_rows<4>(a, s);
    if (a.M <= 8) return launch_rows<8>(a, s);
    return launch_rows<16>(a, s);
}

}  // namespace gemm_f32

// Products with a short B (N up to 16 columns) against a large A: the mirror
// case, bound by reading A once.  Each warp computes whole rows of C (a
// grid-stride loop over rows): its lanes stream the row of A with 16-byte
// loads (512 contiguous bytes a step, four steps in flight), take B's rows for
// their k through L1 (B is K x N, small), keep NR FP32 sums each, and add the
// 32 lanes' sums in a fixed butterfly order.  Every output is summed in one
// order, run after run.
namespace gemm_f32 {
namespace {

constexpr int kColsThreads = 256;
constexpr int kColsUnroll = 4;

template <int NR>
__global__ void __launch_bounds__(kColsThreads)
cols_kernel(const float* __restrict__ A, int64_t lda, const float* __restrict__ B, int64_t ldb,
            float* __restrict__ C, int64_t ldc, int64_t M, int64_t N, int64_t K, int vec_a)
{
    const int lane = threadIdx.x & 31;
    const int64_t wpb = kColsThreads / 32;
    for (int64_t i = (int64_t)blockIdx.x * wpb + threadIdx.x / 32; i < M; i += (int64_t)gridDim.x * wpb) {
        const float* arow = A + i * lda;
        float acc[NR];
#pragma unroll
        for (int j = 0; j < NR; ++j) acc[j] = 0.f;
        for (int64_t k0 = 4 * lane; k0 < K; k0 += 128 * kColsUnroll) {
            float a[kColsUnroll][4];
#pragma unroll
            for (int u = 0; u < kColsUnroll; ++u) {
                const int64_t k = k0 + 128 * u;
                if (vec_a && k + 3 < K) {
                    const float4 v = __ldg(reinterpret_cast<const float4*>(arow + k));
                    a[u][0] = v.x; a[u][1] = v.y; a[u][2] = v.z; a[u][3] = v.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) a[u][c] = k + c < K ? __ldg(arow + k + c) : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kColsUnroll; ++u)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int64_t k = k0 + 128 * u + c;
                    if (k < K) {
                        const float* brow = B + k * ldb;
#pragma unroll
                        for (int j = 0; j < NR; ++j)
                            if (j < N) acc[j] = fmaf(a[u][c], __ldg(brow + j), acc[j]);
                    }
                }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int j = 0; j < NR; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < NR; ++j)
                if (j < N) C[i * ldc + j] = acc[j];
    }
}

template <int NR>
cudaError_t launch_cols(const ColsArgs& a, int sms, cudaStream_t s)
{
    const int64_t wpb = kColsThreads / 32;
    int64_t blocks = (a.M + wpb - 1) / wpb;
    const int64_t cap = (int64_t)sms * 16;
    if (blocks > cap) blocks = cap;
    const int vec_a = (a.lda % 4 == 0) && (reinterpret_cast<uintptr_t>(a.A) % 16 == 0);
    cols_kernel<NR><<<(unsigned)blocks, kColsThreads, 0, s>>>(a.A, a.lda, a.B, a.ldb, a.C, a.ldc, a.M, a.N, a.K,
                                                              vec_a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t cols_launch(const ColsArgs& a, int sms, cudaStream_t s)
{
    if (a.M < 1 || a.N < 1 || a.N > kColsMaxN || a.K < 1 || sms < 1) return cudaErrorInvalidValue;
    if (a.N <= 1) return launch_cols<1>(a, sms, s);
    if (a.N <= 2) return launch_cols<2>(a, sms, s);
    if (a.N <= 4) return launch_cols<4>(a, sms, s);
    if (a.N <= 8) return launch_cols<8>(a, sms, s);
    return launch_cols<16>(a, sms, s);
}

}  // namespace gemm_f32
