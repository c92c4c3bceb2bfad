// tcgen05 3xTF32 GEMM: TMA producer warp, N-stage mbarrier ring, MMA warp
// accumulating in TMEM, epilogue warpgroup.
//
// The pages' double-buffered K-loop ("Double Buffering" technique page and
// "Case Study: The Double-Buffered GEMM") prefetches tile l+1 while computing
// tile l, with one barrier per iteration that means both "the prefetch landed"
// and "everyone is done with the buffer about to be overwritten".  Their
// platform has no copy engine, so the overlap there is only instruction-level.
// On sm_103a the copy engine is real: one thread of a producer warp issues TMA
// bulk-tensor loads into an S-stage shared-memory ring, and the two meanings of
// the pages' single barrier become two mbarriers per stage:
//
//   full[s]   "tile landed"     armed by the producer with the stage's byte
//                               count, completed by the TMA engine;
//   empty[s]  "buffer is free"  completed by tcgen05.commit once the MMAs that
//                               read stage s have finished.
//
// Both A and B of a stage publish through the one full[s] barrier (a single
// expect-tx for all four operand tiles): the coalesced synchronisation of
// "Dependence-aware group synchronization on M1 Max", section "Transformation
// and safety boundary" (copy A; copy B; one fence; MMA), and the WAR hazard
// across the loop back-edge that it keeps is exactly empty[s].
//
// FP32 accuracy from TF32 tensor cores (error-compensated 3xTF32): each operand
// x is split by a pre-pass into hi = RN_tf32(x) and lo = RN_tf32(x - hi), and the
// MMA warp accumulates lo_A*hi_B + hi_A*lo_B + hi_A*hi_B per 8-wide k-step into
// one FP32 TMEM accumulator.  The pre-pass also transposes B to K-major and pads
// K to a multiple of 32, so the tensor maps of the split operands always meet
// TMA's 16-byte rules, whatever the caller's leading dimensions.
//
// Kernel roles (192 threads, one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer (one elected thread)
//   warp 1      TMEM allocator + MMA issuer (one thread)
//   warps 2..5  epilogue: tcgen05.ld TMEM -> registers -> guarded 16-byte stores;
//               warp w reads TMEM lanes 32*(w%4) .. +31 (= tile rows).
// The accumulator is double-buffered in TMEM so the epilogue of one tile runs
// under the main loop of the next.  Every wait is bounded: when a limit runs
// out the thread records a timeout in the status word, all roles leave their
// loops, in-flight copies and MMAs are drained (again with a limit) and TMEM is
// freed before the CTA exits.
#include <cstdint>
#include <cstdio>

#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gemm_f32 {
namespace {

constexpr int kBM = 128;      // tile rows = TMEM lanes
constexpr int kBK = 32;       // fp32 elements per 128-byte swizzle row
constexpr int kUmmaK = 8;     // K of one kind::tf32 MMA
constexpr int kThreads = 192;
constexpr int64_t kDefaultTimeout = int64_t(1) << 32;  // SM clock cycles

struct TcArgs {
    int64_t M, N;
    int64_t ldc, ldp;
    float* C;
    float* partial;
    int* status;
    int64_t timeout;
    int tiles_m, tiles_n;
    int num_kb;          // k-blocks of 32 in the padded K
    int kb_per_split;
    int split_k;
    int terms;           // 3 = 3xTF32, 1 = hi*hi only
    int withhold;        // test hook: 1-based fill index the producer skips (0 = none)
};

// ---------------------------------------------------------------------------
// Operand split pre-pass.
// ---------------------------------------------------------------------------

// Round an FP32 value to the nearest TF32 value (10 explicit mantissa bits),
// ties to even, by integer arithmetic on the bit pattern; the low 13 bits of
// the result are zero.  Inf stays Inf; NaN stays NaN.
__device__ __forceinline__ float tf32_rne(float x)
{
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7F800000u) != 0x7F800000u) u += 0x0FFFu + ((u >> 13) & 1u);
    return __uint_as_float(u & 0xFFFFE000u);
}

__device__ __forceinline__ void split3(float x, float& hi, float& lo)
{
    hi = tf32_rne(x);
    lo = tf32_rne(x - hi);  // x - hi is exact in FP32
}

// A (M x K, lda) -> a_hi, a_lo (M x kp, K-major, zero for k >= K).
__global__ void __launch_bounds__(256)
split_a_kernel(const float* __restrict__ A, int64_t M, int64_t K, int64_t lda, int64_t kp,
               float4* __restrict__ hi, float4* __restrict__ lo, int vec)
{
    const int64_t kp4 = kp / 4;
    const int64_t total = M * kp4;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / kp4, k = (idx % kp4) * 4;
        const float* row = A + i * lda;
        float v[4];
        if (vec && k + 3 < K) {
            const float4 t = __ldg(reinterpret_cast<const float4*>(row + k));
            v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = (k + j < K) ? __ldg(row + k + j) : 0.f;
        }
        float h[4], l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) split3(v[j], h[j], l[j]);
        hi[idx] = make_float4(h[0], h[1], h[2], h[3]);
        lo[idx] = make_float4(l[0], l[1], l[2], l[3]);
    }
}

// B (K x N, ldb) -> b_hi, b_lo (N x kp, i.e. B transposed, K-major), through a
// 32x32 shared-memory tile so both the read (along n) and the write (along k)
// are coalesced.  Grid: x over the kp/32 k-blocks, y strides over n-blocks.
__global__ void __launch_bounds__(256)
split_bt_kernel(const float* __restrict__ B, int64_t K, int64_t N, int64_t ldb, int64_t kp,
                float* __restrict__ hi, float* __restrict__ lo)
{
    __shared__ float tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const int64_t k0 = (int64_t)blockIdx.x * 32;
    for (int64_t n0 = (int64_t)blockIdx.y * 32; n0 < N; n0 += (int64_t)gridDim.y * 32) {
#pragma unroll
        for (int r = ty; r < 32; r += 8) {
            const int64_t k = k0 + r, n = n0 + tx;
            tile[r][tx] = (k < K && n < N) ? __ldg(B + k * ldb + n) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int r = ty; r < 32; r += 8) {
            const int64_t n = n0 + r, k = k0 + tx;
            if (n < N) {
                float h, l;
                split3(tile[tx][r], h, l);
                hi[n * kp + k] = h;
                lo[n * kp + k] = l;
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Main kernel.
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor (tcgen05 format) for a K-major operand tile
// in the 128-byte swizzled layout TMA writes: rows of 128 B, 8-row atoms 1024 B
// apart (stride byte offset), leading byte offset unused for swizzled K-major.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4)
         | ((uint64_t)1 << 16)                  // leading byte offset (unused)
         | ((uint64_t)(1024 >> 4) << 32)        // stride byte offset
         | ((uint64_t)1 << 46)                  // descriptor version (tcgen05)
         | ((uint64_t)2 << 61);                 // swizzle: 128 B
}

// Instruction descriptor, kind::tf32: D fp32, A and B tf32, both K-major,
// M = 128, N = BN.
template <int BN>
__host__ __device__ constexpr uint32_t idesc_tf32()
{
    return (1u << 4)                 // D format: F32
         | (2u << 7)                 // A format: TF32
         | (2u << 10)                // B format: TF32
         | ((uint32_t)(BN >> 3) << 17)
         | ((uint32_t)(kBM >> 4) << 24);
}

template <int BN, int STAGES>
struct TcLayout {
    static constexpr int A_BYTES = kBM * kBK * 4;   // 16 KB
    static constexpr int B_BYTES = BN * kBK * 4;
    static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int BAR_BYTES = 8 * (2 * STAGES + 5) + 16;
    static constexpr int SMEM_BYTES = 1024 + RING_BYTES + BAR_BYTES;
    static constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulator buffers
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS >= 32 && TMEM_COLS <= 512, "TMEM cols");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Bounded wait on phase `parity` of an mbarrier.  Gives up when the limit runs
// out or another role has raised the abort flag; on a timeout it records the
// status word and raises the flag.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, int64_t limit,
                                           volatile int* abort_flag, int* status)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            atomicExch(status, kStatusTimeout);
            *abort_flag = 1;
            return false;
        }
    }
}

// Tile order: groups of 8 tile-rows, column-major inside a group, so the CTAs
// running together share A and B panels in L2.
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int& tm, int& tn)
{
    constexpr int G = 8;
    const int group_size = G * tiles_n;
    const int gid = tile / group_size;
    const int first_m = gid * G;
    const int gsz = min(tiles_m - first_m, G);
    const int r = tile % group_size;
    tm = first_m + r % gsz;
    tn = r / gsz;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_ahi, const __grid_constant__ CUtensorMap tm_alo,
               const __grid_constant__ CUtensorMap tm_bhi, const __grid_constant__ CUtensorMap tm_blo,
               const TcArgs args)
{
    using L = TcLayout<BN, STAGES>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Align the ring to 1024 B (128-byte swizzle atoms).
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t ring = (raw_addr + 1023u) & ~1023u;
    uint8_t* ring_ptr = smem_raw + (ring - raw_addr);
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring_ptr + L::RING_BYTES);
    // bars[0..S-1] full, [S..2S-1] empty, [2S..2S+1] tmem_full, [2S+2..2S+3] tmem_empty,
    // [2S+4] drain; then the TMEM base address slot and the abort flag.
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto full_bar = [&](int s) { return ptx::smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return ptx::smem_u32(bars + STAGES + s); };
    auto tfull_bar = [&](int b) { return ptx::smem_u32(bars + 2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return ptx::smem_u32(bars + 2 * STAGES + 2 + b); };
    const uint32_t drain_bar = ptx::smem_u32(bars + 2 * STAGES + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), 4);
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tm_ahi);
        ptx::tma_prefetch_desc(&tm_alo);
        ptx::tma_prefetch_desc(&tm_bhi);
        ptx::tma_prefetch_desc(&tm_blo);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), L::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_tiles = args.tiles_m * args.tiles_n;
    const int num_work = num_tiles * args.split_k;
    const int64_t limit = args.timeout;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t fills = 0;
            bool stop = false;
            for (int w = blockIdx.x; w < num_work && !stop; w += gridDim.x) {
                const int z = w / num_tiles;
                int tm, tn;
                tile_coords(w % num_tiles, args.tiles_m, args.tiles_n, tm, tn);
                const int kb0 = z * args.kb_per_split;
                const int kb1 = min(args.num_kb, kb0 + args.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(empty_bar(stage), phase ^ 1u, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
                    ++fills;
                    if (fills != (uint32_t)args.withhold) {
                        const uint32_t sb = ring + stage * L::STAGE_BYTES;
                        ptx::mbar_arrive_expect_tx(full_bar(stage), L::STAGE_BYTES);
                        const int kc = kb * kBK;
                        ptx::tma_load_2d(sb, &tm_ahi, full_bar(stage), kc, tm * kBM);
                        ptx::tma_load_2d(sb + L::A_BYTES, &tm_alo, full_bar(stage), kc, tm * kBM);
                        ptx::tma_load_2d(sb + 2 * L::A_BYTES, &tm_bhi, full_bar(stage), kc, tn * BN);
                        ptx::tma_load_2d(sb + 2 * L::A_BYTES + L::B_BYTES, &tm_blo, full_bar(stage), kc,
                                         tn * BN);
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Drain: the last fill of every slot must have landed before the CTA
            // may exit (a withheld fill was never armed and is skipped).
            const uint32_t total = fills;
            for (int s = 0; s < STAGES; ++s) {
                if ((uint32_t)s >= total) break;
                const uint32_t last = (total - 1 - s) / STAGES * STAGES + s;  // index of last fill of slot s
                if (last + 1 == (uint32_t)args.withhold) continue;
                const uint32_t par = (last / STAGES) & 1u;
                const long long t0 = clock64();
                while (!ptx::mbar_try_wait(full_bar(s), par)) {
                    if (clock64() - t0 > limit) { atomicExch(args.status, kStatusTimeout); break; }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_tf32<BN>();
            int stage = 0;
            uint32_t phase = 0;
            int iter = 0;
            bool stop = false;
            for (int w = blockIdx.x; w < num_work && !stop; w += gridDim.x, ++iter) {
                const int z = w / num_tiles;
                const int kb0 = z * args.kb_per_split;
                const int kb1 = min(args.num_kb, kb0 + args.kb_per_split);
                const int buf = iter & 1;
                const uint32_t tphase = (iter >> 1) & 1;
                if (!wait_phase(tempty_bar(buf), tphase ^ 1u, limit, abort_flag, args.status)) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(full_bar(stage), phase, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sb = ring + stage * L::STAGE_BYTES;
                    const uint32_t a_hi = sb, a_lo = sb + L::A_BYTES;
                    const uint32_t b_hi = sb + 2 * L::A_BYTES, b_lo = b_hi + L::B_BYTES;
#pragma unroll
                    for (int ks = 0; ks < kBK / kUmmaK; ++ks) {
                        const uint32_t off = ks * kUmmaK * 4;  // 32 B along the swizzled row
                        const uint32_t acc = (kb > kb0 || ks > 0) ? 1u : 0u;
                        if (args.terms == 3) {
                            ptx::mma_tf32(d_tmem, sw128_desc(a_lo + off), sw128_desc(b_hi + off), idesc, acc);
                            ptx::mma_tf32(d_tmem, sw128_desc(a_hi + off), sw128_desc(b_lo + off), idesc, 1u);
                            ptx::mma_tf32(d_tmem, sw128_desc(a_hi + off), sw128_desc(b_hi + off), idesc, 1u);
                        } else {
                            ptx::mma_tf32(d_tmem, sw128_desc(a_hi + off), sw128_desc(b_hi + off), idesc, acc);
                        }
                    }
                    ptx::mma_commit(empty_bar(stage));  // slot free once these MMAs finish
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (stop) break;
                ptx::mma_commit(tfull_bar(buf));  // accumulator complete
            }
            // Drain every MMA this thread issued before TMEM is released.
            ptx::mma_commit(drain_bar);
            const long long t0 = clock64();
            while (!ptx::mbar_try_wait(drain_bar, 0)) {
                if (clock64() - t0 > limit) { atomicExch(args.status, kStatusTimeout); break; }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------ epilogue ------------------------------
        const int quad = warp & 3;              // TMEM lane quadrant this warp may access
        const int row_in_tile = quad * 32 + lane;
        int iter = 0;
        for (int w = blockIdx.x; w < num_work; w += gridDim.x, ++iter) {
            const int z = w / num_tiles;
            int tm, tn;
            tile_coords(w % num_tiles, args.tiles_m, args.tiles_n, tm, tn);
            const int buf = iter & 1;
            const uint32_t tphase = (iter >> 1) & 1;
            if (!wait_phase(tfull_bar(buf), tphase, limit, abort_flag, args.status)) break;
            ptx::tc_fence_after();
            float* out;
            int64_t ld;
            bool vec;
            if (args.split_k > 1) {
                out = args.partial + (int64_t)z * args.M * args.ldp;
                ld = args.ldp;
                vec = true;
            } else {
                out = args.C;
                ld = args.ldc;
                vec = ((ld & 3) == 0) && ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
            }
            const int64_t grow = (int64_t)tm * kBM + row_in_tile;
            const bool row_ok = grow < args.M;
            float* orow = out + (row_ok ? grow : 0) * ld;
            const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + buf * BN;
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
                uint32_t r[16];
                ptx::tmem_ld_32x32b_x16(taddr + c, r);
                ptx::tmem_wait_ld();
                const int64_t gn = (int64_t)tn * BN + c;
                if (row_ok) {
                    if (vec && gn + 15 < args.N) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4*>(orow + gn + j) =
                                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (gn + j < args.N) orow[gn + j] = __uint_as_float(r[j]);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty_bar(buf));
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

EncodeFn get_encode()
{
    static EncodeFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    }
    return fn;
}

// 2-D tensor map over a rows x kp K-major FP32 buffer, box {32, box_rows},
// 128-byte swizzle, zero fill outside.
cudaError_t encode_kmajor(void* out, float* base, int64_t rows, int64_t kp, int box_rows)
{
    EncodeFn enc = get_encode();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)kp, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(kp * 4)};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int BN, int STAGES>
cudaError_t launch_main(const TcPlanState& st, const TcArgs& a, cudaStream_t s)
{
    using L = TcLayout<BN, STAGES>;
    auto kern = tc_gemm_kernel<BN, STAGES>;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int work = a.tiles_m * a.tiles_n * a.split_k;
    const int grid = work < st.num_sms ? work : st.num_sms;
    kern<<<grid, kThreads, L::SMEM_BYTES, s>>>(
        *reinterpret_cast<const CUtensorMap*>(st.tmap_a_hi), *reinterpret_cast<const CUtensorMap*>(st.tmap_a_lo),
        *reinterpret_cast<const CUtensorMap*>(st.tmap_b_hi), *reinterpret_cast<const CUtensorMap*>(st.tmap_b_lo), a);
    return cudaGetLastError();
}

using MainFn = cudaError_t (*)(const TcPlanState&, const TcArgs&, cudaStream_t);
struct TcEntry {
    TcConfig cfg;
    MainFn fn;
};
const TcEntry kTc[] = {
    {{128, 128, 32, 3}, launch_main<128, 3>},
    {{128, 256, 32, 2}, launch_main<256, 2>},
    {{128, 64, 32, 4}, launch_main<64, 4>},
};

int grid_cap(int64_t work, int sms)
{
    const int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

int tc_num_configs() { return (int)(sizeof(kTc) / sizeof(kTc[0])); }
const TcConfig& tc_config(int id) { return kTc[id].cfg; }
int tc_find_config(int bn, int stages)
{
    for (int i = 0; i < tc_num_configs(); ++i)
        if (kTc[i].cfg.bn == bn && kTc[i].cfg.stages == stages) return i;
    // Stage count not compiled for this tile width: take the one that is.
    if (stages == 0)
        for (int i = 0; i < tc_num_configs(); ++i)
            if (kTc[i].cfg.bn == bn) return i;
    return -1;
}

cudaError_t tc_prepare(TcPlanState& st, int64_t M, int64_t N, int64_t K)
{
    (void)K;
    const TcConfig& c = kTc[st.config_id].cfg;
    cudaError_t e;
    if ((e = encode_kmajor(st.tmap_a_hi, st.a_hi, M, st.kp, kBM)) != cudaSuccess) return e;
    if ((e = encode_kmajor(st.tmap_a_lo, st.a_lo, M, st.kp, kBM)) != cudaSuccess) return e;
    if ((e = encode_kmajor(st.tmap_b_hi, st.b_hi, N, st.kp, c.bn)) != cudaSuccess) return e;
    if ((e = encode_kmajor(st.tmap_b_lo, st.b_lo, N, st.kp, c.bn)) != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t tc_launch(const TcPlanState& st, int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                      const float* B, int64_t ldb, float* C, int64_t ldc, int* status, cudaStream_t s,
                      cudaEvent_t* ev)
{
    const TcConfig& c = kTc[st.config_id].cfg;
    if (ev) cudaEventRecord(ev[0], s);
    // 1. Split the operands (and transpose B) into the plan's scratch.
    {
        const int vec = (lda % 4 == 0) && (reinterpret_cast<uintptr_t>(A) % 16 == 0);
        split_a_kernel<<<grid_cap(M * (st.kp / 4), st.num_sms), 256, 0, s>>>(
            A, M, K, lda, st.kp, reinterpret_cast<float4*>(st.a_hi), reinterpret_cast<float4*>(st.a_lo), vec);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const int64_t nb = (N + 31) / 32;
        dim3 g((unsigned)(st.kp / 32), (unsigned)(nb < 65535 ? nb : 65535));
        split_bt_kernel<<<g, 256, 0, s>>>(B, K, N, ldb, st.kp, st.b_hi, st.b_lo);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // 2. The pipelined tensor-core GEMM.
    TcArgs a{};
    a.M = M; a.N = N; a.ldc = ldc; a.ldp = st.ldp; a.C = C; a.partial = st.partial;
    a.status = status;
    a.timeout = st.timeout_cycles > 0 ? st.timeout_cycles : kDefaultTimeout;
    a.tiles_m = (int)((M + kBM - 1) / kBM);
    a.tiles_n = (int)((N + c.bn - 1) / c.bn);
    a.num_kb = (int)(st.kp / kBK);
    a.split_k = st.split_k;
    a.kb_per_split = st.kb_per_split;
    a.terms = st.terms;
    a.withhold = st.withhold_stage;
    if (ev) cudaEventRecord(ev[1], s);
    cudaError_t e = kTc[st.config_id].fn(st, a, s);
    if (e != cudaSuccess) return e;
    if (ev) cudaEventRecord(ev[2], s);
    // 3. Deterministic split-K sum.
    if (st.split_k > 1) e = splitk_reduce_launch(st.partial, st.split_k, M, N, st.ldp, C, ldc, s);
    if (ev) cudaEventRecord(ev[3], s);
    return e;
}

}  // namespace gemm_f32
