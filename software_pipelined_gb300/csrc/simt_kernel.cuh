// SIMT FFMA GEMM kernel template (instantiated in simt_configs_*.cu).
//
// This is the pages' software-pipelined K-loop ("Double Buffering" technique
// page; "Case Study: The Double-Buffered GEMM") on GB300's per-thread async
// copy: every thread issues the cp.async prefetch of tile l+S-1 and then
// computes on tile l, so the copy engine and the FFMA pipe overlap.  With S=2
// it is exactly the double-buffered loop: one __syncthreads per iteration does
// the pages' "double duty" (tile l has landed for every thread, and every thread
// has finished reading the buffer about to be refilled).  S=1 is the
// single-buffered sibling (load, barrier, compute, barrier) kept for the
// pipeline-depth ablation.
//
// SEP = true is the ablation of the barrier coalescing of "Dependence-aware
// group synchronization on M1 Max" ("Transformation and safety boundary"): A
// and B are copied as separate cp.async groups and each gets its own barrier
// (copy A; barrier; copy B; barrier; compute; ...), where the default form
// publishes both with one barrier.
//
// KSL > 1 splits K inside the CTA ("sliced K"): KSL groups of threads share
// the staged tiles, group g taking k = g*BK/KSL .. (g+1)*BK/KSL-1 of every
// K-tile with its own register tile; at the end groups 1..KSL-1 hand their
// tiles to group 0 through shared memory, which adds them in group order and
// stores.  For small grids (tens of CTAs) it multiplies the warps an SM can
// switch between without a second (reduction) launch.
//
// Layout: A tile As[BM][BK+4] (row-major, as in global memory, so the copy is a
// straight 16-byte cp.async when rows are 16-byte aligned), B tile
// Bs[BK][BN+4].  An operand whose rows are not 16-byte aligned (VA / VB false:
// a leading dimension that is not a multiple of 4, or a base off a 16-byte
// boundary) is staged through registers in the steady state: each thread loads 4
// consecutive floats of a row (four 4-byte loads, consecutive threads on
// consecutive chunks) and writes them with one 16-byte shared store.  In the
// multi-stage loop those loads of tile t+S-1 are issued before tile t's FFMAs
// and their shared stores follow them, so the copy still overlaps the math;
// the prologue's tiles go by 4-byte cp.async, all in flight at once.
// Each thread owns a TM x TN register tile built from 4x4 blocks
// spread BM/(TM/4) rows and BN/(TN/4) columns apart, so that a warp's 16-byte
// fragment loads hit distinct banks.  A fragments are read as float4 along k
// (4 k-steps per load), B fragments as float4 along n: lanes that need the
// same float4 read the same address, which shared memory broadcasts.  SHF is
// the alternative of the task statement's "warp-shuffle fragment loads" (an
// ablation): each distinct float4 a warp needs is read by one lane and handed
// to the others with shuffles.
#pragma once
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace gemm_f32 {
namespace simt_detail {

template <int BM, int BN, int BK, int TM, int TN, int STAGES, bool VA, bool VB, bool SEP, int KSL, bool SHF>
struct SimtKernel {
    static constexpr int TX = BN / TN;
    static constexpr int TY = BM / TM;
    static constexpr int NT = TX * TY;       // threads of one K-slice group
    static constexpr int NTT = NT * KSL;     // threads of the CTA
    static constexpr int LDA_S = BK + 4;   // floats per As row
    static constexpr int LDB_S = BN + 4;   // floats per Bs row
    static constexpr int A_STAGE = BM * LDA_S;
    static constexpr int B_STAGE = BK * LDB_S;
    static constexpr int RING_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
    static constexpr int RED_BYTES = (KSL - 1) * NT * TM * TN * 4;  // the groups' hand-over
    static constexpr int SMEM_BYTES = RING_BYTES > RED_BYTES ? RING_BYTES : RED_BYTES;
    static_assert(TM % 4 == 0 && TN % 4 == 0, "register tile is built from 4x4 blocks");
    static_assert(BK % (4 * KSL) == 0, "each K-slice group takes whole float4 columns of A");
    static_assert(NT >= 32 && NTT <= 1024, "block size");
    static_assert(!SEP || STAGES <= 2, "separate barriers: 1 or 2 stages");
    static_assert(!SEP || KSL == 1, "the barrier ablation runs unsliced");
    static_assert(!SHF || (32 % TX == 0 && (32 / TX) * TM <= 32 && BN / 4 <= 32 && NT % 32 == 0),
                  "shuffle fragments: a warp's distinct float4 fit its lanes");
    // chunks of 4 floats per tile, and per thread when staged through registers
    static constexpr int A_CH = BM * BK / 4;
    static constexpr int B_CH = BK * BN / 4;
    static constexpr int RA = VA ? 1 : (A_CH + NTT - 1) / NTT;
    static constexpr int RB = VB ? 1 : (B_CH + NTT - 1) / NTT;
};

template <int BM, int BN, int BK, int TM, int TN, int STAGES, bool VA, bool VB, bool SEP, int KSL, bool SHF>
__global__ void __launch_bounds__((BM / TM) * (BN / TN) * KSL)
simt_gemm_kernel(SimtArgs a)
{
    using KT = SimtKernel<BM, BN, BK, TM, TN, STAGES, VA, VB, SEP, KSL, SHF>;
    constexpr int NT = KT::NT, NTT = KT::NTT, TX = KT::TX;
    constexpr int RG = TM / 4, CG = TN / 4;
    extern __shared__ __align__(16) float smem[];
    float* As = smem;
    float* Bs = smem + STAGES * KT::A_STAGE;

    const int tid = threadIdx.x;              // copies: all NTT threads
    const int slice = tid / NT;               // K-slice group
    const int tt = tid % NT;                  // thread within the group
    const int tx = tt % TX, ty = tt / TX;
    const int64_t m0 = (int64_t)blockIdx.y * BM;
    const int64_t n0 = (int64_t)blockIdx.x * BN;
    const bool batched = a.batch > 1;
    const int64_t kbeg = batched ? 0 : (int64_t)blockIdx.z * a.k_chunk;
    const int64_t kend = batched ? a.K : min(a.K, kbeg + a.k_chunk);
    const int nk = kend > kbeg ? (int)((kend - kbeg + BK - 1) / BK) : 0;
    const int64_t M = a.M, N = a.N;
    const float* __restrict__ A = a.A + (batched ? (int64_t)blockIdx.z * a.stride_a : 0);
    const float* __restrict__ B = a.B + (batched ? (int64_t)blockIdx.z * a.stride_b : 0);
    // Programmatic serialisation: wait for the previous kernel's writes before
    // the first copy (a no-op when launched without the attribute).
    asm volatile("griddepcontrol.wait;\n" ::: "memory");

    // Register staging of the operands whose rows are not 16-byte aligned:
    // chunk c of a tile is 4 consecutive floats of one row; out-of-range
    // elements (ragged M, N or K) are zeros.
    float4 ra[KT::RA], rb[KT::RB];
    auto gather_a = [&](int t) {
        const int64_t k0 = kbeg + (int64_t)t * BK;
#pragma unroll
        for (int i = 0; i < KT::RA; ++i) {
            const int c = tid + i * NTT;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (c < KT::A_CH) {
                const int r = c / (BK / 4), kc = (c % (BK / 4)) * 4;
                const int64_t gm = m0 + r, gk = k0 + kc;
                if (gm < M) {
                    const float* p = A + gm * a.lda + gk;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (gk + j < kend) v[j] = __ldg(p + j);
                }
            }
            ra[i] = make_float4(v[0], v[1], v[2], v[3]);
        }
    };
    auto put_a = [&](int st) {
        float* as = As + st * KT::A_STAGE;
#pragma unroll
        for (int i = 0; i < KT::RA; ++i) {
            const int c = tid + i * NTT;
            if (c < KT::A_CH)
                *reinterpret_cast<float4*>(as + (c / (BK / 4)) * KT::LDA_S + (c % (BK / 4)) * 4) = ra[i];
        }
    };
    auto gather_b = [&](int t) {
        const int64_t k0 = kbeg + (int64_t)t * BK;
#pragma unroll
        for (int i = 0; i < KT::RB; ++i) {
            const int c = tid + i * NTT;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (c < KT::B_CH) {
                const int r = c / (BN / 4), nc = (c % (BN / 4)) * 4;
                const int64_t gk = k0 + r, gn = n0 + nc;
                if (gk < kend) {
                    const float* p = B + gk * a.ldb + gn;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (gn + j < N) v[j] = __ldg(p + j);
                }
            }
            rb[i] = make_float4(v[0], v[1], v[2], v[3]);
        }
    };
    auto put_b = [&](int st) {
        float* bs = Bs + st * KT::B_STAGE;
#pragma unroll
        for (int i = 0; i < KT::RB; ++i) {
            const int c = tid + i * NTT;
            if (c < KT::B_CH)
                *reinterpret_cast<float4*>(bs + (c / (BN / 4)) * KT::LDB_S + (c % (BN / 4)) * 4) = rb[i];
        }
    };

    // Copies of K-tile t into ring slot st, all by cp.async (out-of-range
    // elements zero-filled by the copy itself): 16 bytes at a time for 16-byte
    // aligned rows, else four 4-byte copies per chunk of 4 floats.  These serve
    // the prologue (every tile of it in flight at once) and the single-stage
    // and barrier-ablation loops; the multi-stage loop stages unaligned rows
    // through registers instead (gather / put), which measured faster there.
    auto load_a = [&](int st, int t) {
        const int64_t k0 = kbeg + (int64_t)t * BK;
        float* as = As + st * KT::A_STAGE;
        if constexpr (VA) {
            for (int c = tid; c < BM * BK / 4; c += NTT) {
                const int r = c / (BK / 4), kc = (c % (BK / 4)) * 4;
                const int64_t gm = m0 + r, gk = k0 + kc;
                int bytes = 0;
                const float* src = A;
                if (gm < M && gk < kend) {
                    bytes = 4 * (int)(kend - gk < 4 ? kend - gk : 4);
                    src = A + gm * a.lda + gk;
                }
                ptx::cp_async_16(ptx::smem_u32(as + r * KT::LDA_S + kc), src, bytes);
            }
        } else {
            for (int c = tid; c < KT::A_CH; c += NTT) {
                const int r = c / (BK / 4), kc = (c % (BK / 4)) * 4;
                const int64_t gm = m0 + r, gk = k0 + kc;
                const uint32_t d = ptx::smem_u32(as + r * KT::LDA_S + kc);
                const float* p = A + (gm < M ? gm : 0) * a.lda + gk;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool ok = gm < M && gk + j < kend;
                    ptx::cp_async_4(d + 4 * j, ok ? p + j : A, ok ? 4 : 0);
                }
            }
        }
    };
    auto load_b = [&](int st, int t) {
        const int64_t k0 = kbeg + (int64_t)t * BK;
        float* bs = Bs + st * KT::B_STAGE;
        if constexpr (VB) {
            for (int c = tid; c < BK * BN / 4; c += NTT) {
                const int r = c / (BN / 4), nc = (c % (BN / 4)) * 4;
                const int64_t gk = k0 + r, gn = n0 + nc;
                int bytes = 0;
                const float* src = B;
                if (gk < kend && gn < N) {
                    bytes = 4 * (int)(N - gn < 4 ? N - gn : 4);
                    src = B + gk * a.ldb + gn;
                }
                ptx::cp_async_16(ptx::smem_u32(bs + r * KT::LDB_S + nc), src, bytes);
            }
        } else {
            for (int c = tid; c < KT::B_CH; c += NTT) {
                const int r = c / (BN / 4), nc = (c % (BN / 4)) * 4;
                const int64_t gk = k0 + r, gn = n0 + nc;
                const uint32_t d = ptx::smem_u32(bs + r * KT::LDB_S + nc);
                const float* p = B + (gk < kend ? gk : 0) * a.ldb + gn;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool ok = gk < kend && gn + j < N;
                    ptx::cp_async_4(d + 4 * j, ok ? p + j : B, ok ? 4 : 0);
                }
            }
        }
    };
    auto load_tile = [&](int st, int t) {
        load_a(st, t);
        load_b(st, t);
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    // Shuffle fragments: this warp's first thread-grid row, and the float4
    // each lane reads for the warp (A: row w*TM + i of the warp's WR x TM rows;
    // B: column chunk h*TX + x of the BN/4 chunks).
    constexpr int WR = SHF ? 32 / TX : 1;
    const int lane = tt & 31;
    const int ty0 = (tt & ~31) / TX;
    auto shfl4 = [](const float4& v, int src) {
        return make_float4(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src),
                           __shfl_sync(0xffffffffu, v.z, src), __shfl_sync(0xffffffffu, v.w, src));
    };
    const int a_row_of_lane = ((lane % TM) / 4) * (BM / RG) + (ty0 + lane / TM) * 4 + (lane % 4);
    const int b_col_of_lane = (lane / TX) * (BN / CG) + (lane % TX) * 4;

    auto compute_tile = [&](int st) {
        const float* as = As + st * KT::A_STAGE;
        const float* bs = Bs + st * KT::B_STAGE;
#pragma unroll
        for (int k4 = 0; k4 < BK / KSL; k4 += 4) {
            const int kk = slice * (BK / KSL) + k4;
            float4 av[TM];
            if constexpr (SHF) {
                float4 mine = make_float4(0.f, 0.f, 0.f, 0.f);
                if (lane < WR * TM) mine = *reinterpret_cast<const float4*>(as + a_row_of_lane * KT::LDA_S + kk);
#pragma unroll
                for (int i = 0; i < TM; ++i) av[i] = shfl4(mine, (ty - ty0) * TM + i);
            } else {
#pragma unroll
                for (int g = 0; g < RG; ++g)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        av[g * 4 + i] = *reinterpret_cast<const float4*>(
                            as + (g * (BM / RG) + ty * 4 + i) * KT::LDA_S + kk);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float bv[TN];
                if constexpr (SHF) {
                    float4 mine = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (lane < BN / 4) mine = *reinterpret_cast<const float4*>(bs + (kk + q) * KT::LDB_S + b_col_of_lane);
#pragma unroll
                    for (int h = 0; h < CG; ++h) {
                        const float4 t = shfl4(mine, h * TX + tx);
                        bv[h * 4 + 0] = t.x; bv[h * 4 + 1] = t.y;
                        bv[h * 4 + 2] = t.z; bv[h * 4 + 3] = t.w;
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < CG; ++h) {
                        const float4 t = *reinterpret_cast<const float4*>(
                            bs + (kk + q) * KT::LDB_S + h * (BN / CG) + tx * 4);
                        bv[h * 4 + 0] = t.x; bv[h * 4 + 1] = t.y;
                        bv[h * 4 + 2] = t.z; bv[h * 4 + 3] = t.w;
                    }
                }
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const float av_q = q == 0 ? av[i].x : q == 1 ? av[i].y : q == 2 ? av[i].z : av[i].w;
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av_q, bv[j], acc[i][j]);
                }
            }
        }
    };

    if constexpr (SEP && STAGES == 1) {
        // Single-buffered, separate publication: copy A; barrier; copy B;
        // barrier; compute; barrier (three per step).
        for (int t = 0; t < nk; ++t) {
            load_a(0, t);
            ptx::cp_async_commit();
            ptx::cp_async_wait<0>();
            __syncthreads();
            load_b(0, t);
            ptx::cp_async_commit();
            ptx::cp_async_wait<0>();
            __syncthreads();
            compute_tile(0);
            __syncthreads();
        }
    } else if constexpr (SEP) {
        // Double-buffered, separate publication: A and B of a tile are two
        // cp.async groups, each published by its own barrier (two per step).
        load_a(0, 0);
        ptx::cp_async_commit();
        load_b(0, 0);
        ptx::cp_async_commit();
        for (int t = 0; t < nk; ++t) {
            ptx::cp_async_wait<1>();   // A of tile t
            __syncthreads();
            ptx::cp_async_wait<0>();   // B of tile t
            __syncthreads();           // also: everyone is done with slot (t+1)%2
            if (t + 1 < nk) load_a((t + 1) & 1, t + 1);
            ptx::cp_async_commit();
            if (t + 1 < nk) load_b((t + 1) & 1, t + 1);
            ptx::cp_async_commit();
            compute_tile(t & 1);
        }
        ptx::cp_async_wait<0>();
    } else if constexpr (STAGES == 1) {
        // Single-buffered: load, wait, barrier, compute, barrier (two per step).
        for (int t = 0; t < nk; ++t) {
            load_tile(0, t);
            ptx::cp_async_commit();
            ptx::cp_async_wait<0>();
            __syncthreads();
            compute_tile(0);
            __syncthreads();
        }
    } else {
        // Prologue: tiles 0 .. S-2 in flight.
#pragma unroll
        for (int s = 0; s < STAGES - 1; ++s) {
            if (s < nk) load_tile(s, s);
            ptx::cp_async_commit();
        }
        for (int t = 0; t < nk; ++t) {
            ptx::cp_async_wait<STAGES - 2>();  // my copies of tile t have landed
            __syncthreads();                   // everyone's have, and slot (t-1)%S is free
            const int nt = t + STAGES - 1;
            if (nt < nk) {
                // aligned operands: cp.async into the free slot; the others:
                // their loads now, their shared stores after this tile's FFMAs
                // (into the same free slot, published by the next barrier)
                if constexpr (VA) load_a(nt % STAGES, nt); else gather_a(nt);
                if constexpr (VB) load_b(nt % STAGES, nt); else gather_b(nt);
            }
            ptx::cp_async_commit();
            compute_tile(t % STAGES);
            if (nt < nk) {
                if constexpr (!VA) put_a(nt % STAGES);
                if constexpr (!VB) put_b(nt % STAGES);
            }
        }
        ptx::cp_async_wait<0>();
    }
    // The next kernel on the stream may launch its CTAs now, during this
    // epilogue.  Not earlier: waiting CTAs of the next launches (each would
    // release its own successor) would fill the SMs' slots and shared memory
    // while this grid still runs.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    if constexpr (KSL > 1) {
        // Hand the register tiles of groups 1..KSL-1 to group 0 (lane-major:
        // consecutive threads, consecutive words), which adds them in order.
        __syncthreads();  // every group is done reading the ring
        float* red = smem;
        if (slice > 0) {
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) red[((slice - 1) * TM * TN + i * TN + j) * NT + tt] = acc[i][j];
        }
        __syncthreads();
        if (slice > 0) return;
        for (int g = 1; g < KSL; ++g)
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] += red[((g - 1) * TM * TN + i * TN + j) * NT + tt];
    }

    // Epilogue: guarded stores of the register tile (16-byte when aligned).
    float* out;
    int64_t ld;
    bool vec;
    if (a.split_k > 1) {
        out = a.partial + (int64_t)blockIdx.z * M * a.ldp;
        ld = a.ldp;
        vec = true;
    } else {
        out = a.C + (batched ? (int64_t)blockIdx.z * a.stride_c : 0);
        ld = a.ldc;
        vec = ((ld & 3) == 0) && ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int64_t gm = m0 + (i / 4) * (BM / RG) + ty * 4 + (i % 4);
        if (gm >= M) continue;
        float* row = out + gm * ld;
#pragma unroll
        for (int h = 0; h < CG; ++h) {
            const int64_t gn = n0 + h * (BN / CG) + tx * 4;
            if (vec && gn + 3 < N) {
                *reinterpret_cast<float4*>(row + gn) =
                    make_float4(acc[i][h * 4 + 0], acc[i][h * 4 + 1], acc[i][h * 4 + 2], acc[i][h * 4 + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (gn + j < N) row[gn + j] = acc[i][h * 4 + j];
            }
        }
    }
}

template <int BM, int BN, int BK, int TM, int TN, int STAGES, bool VA, bool VB, bool SEP, int KSL, bool SHF>
cudaError_t launch_one(const SimtArgs& a, cudaStream_t s)
{
    using KT = SimtKernel<BM, BN, BK, TM, TN, STAGES, VA, VB, SEP, KSL, SHF>;
    auto kern = simt_gemm_kernel<BM, BN, BK, TM, TN, STAGES, VA, VB, SEP, KSL, SHF>;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = smem_limit_once(kern, KT::SMEM_BYTES, smem_set); e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.N + BN - 1) / BN), (unsigned)((a.M + BM - 1) / BM),
                       (unsigned)(a.batch > 1 ? a.batch : a.split_k));
    cfg.blockDim = dim3(KT::NTT);
    cfg.dynamicSmemBytes = KT::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int BM, int BN, int BK, int TM, int TN, int STAGES, bool SEP = false, int KSL = 1, bool SHF = false>
cudaError_t launch_cfg(const SimtArgs& a, cudaStream_t s)
{
    const bool va = (a.lda % 4 == 0) && (reinterpret_cast<uintptr_t>(a.A) % 16 == 0) &&
                    (a.batch <= 1 || a.stride_a % 4 == 0);
    const bool vb = (a.ldb % 4 == 0) && (reinterpret_cast<uintptr_t>(a.B) % 16 == 0) &&
                    (a.batch <= 1 || a.stride_b % 4 == 0);
    if (va && vb) return launch_one<BM, BN, BK, TM, TN, STAGES, true, true, SEP, KSL, SHF>(a, s);
    if (va) return launch_one<BM, BN, BK, TM, TN, STAGES, true, false, SEP, KSL, SHF>(a, s);
    if (vb) return launch_one<BM, BN, BK, TM, TN, STAGES, false, true, SEP, KSL, SHF>(a, s);
    return launch_one<BM, BN, BK, TM, TN, STAGES, false, false, SEP, KSL, SHF>(a, s);
}

using LaunchFn = cudaError_t (*)(const SimtArgs&, cudaStream_t);
struct SimtEntry {
    SimtConfig cfg;
    LaunchFn fn;
};

}  // namespace simt_detail
}  // namespace gemm_f32
