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
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace gemm_f32 {
namespace {

using namespace tc;
constexpr int kThreads = 192;

// ---------------------------------------------------------------------------
// Operand split pre-pass.
// ---------------------------------------------------------------------------

constexpr int kSplitBK = 32;    // k rows per B tile of the split pre-pass
constexpr int kSplitBN = 128;   // n columns per B tile

// One launch splits both operands.  Blocks [0, a_blocks) stream A (M x K, lda)
// into a_hi, a_lo (M x kp, K-major, zero for k >= K), 16 bytes at a time where
// the rows allow; with a_lo_only they write only lo = A - trunc_tf32(A) rounded
// (the GEMM then reads hi straight from A, truncated by the MMA).  The remaining blocks each take a 32 (k) x 128 (n) tile of B
// (K x N, ldb), stage it in shared memory and write it transposed to b_hi,
// b_lo (N x kp): reads are coalesced along n, writes along k.  The last thing
// each block does is allow the dependent GEMM launch to start its prologue.
__global__ void __launch_bounds__(256)
split_operands_kernel(const float* __restrict__ A, int64_t M, int64_t K, int64_t lda, int vec_a,
                      const float* __restrict__ B, int64_t N, int64_t ldb, int vec_b, int64_t kp,
                      float4* __restrict__ a_hi, float4* __restrict__ a_lo,
                      float* __restrict__ b_hi, float* __restrict__ b_lo, int a_blocks, int a_lo_only)
{
    if ((int)blockIdx.x < a_blocks) {
        const int64_t kp4 = kp / 4;
        const int64_t total = M * kp4;
        for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
             idx += (int64_t)a_blocks * blockDim.x) {
            const int64_t i = idx / kp4, k = (idx % kp4) * 4;
            const float* row = A + i * lda;
            float v[4];
            if (vec_a && k + 3 < K) {
                const float4 t = __ldg(reinterpret_cast<const float4*>(row + k));
                v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = (k + j < K) ? __ldg(row + k + j) : 0.f;
            }
            if (a_lo_only) {
                // hi_A is the caller's A itself (the MMA truncates it): only lo
                a_lo[idx] = make_float4(lo_part(v[0]), lo_part(v[1]), lo_part(v[2]), lo_part(v[3]));
                continue;
            }
            float h[4], l[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) split3(v[j], h[j], l[j]);
            a_hi[idx] = make_float4(h[0], h[1], h[2], h[3]);
            a_lo[idx] = make_float4(l[0], l[1], l[2], l[3]);
        }
    } else {
        __shared__ float tile[kSplitBK][kSplitBN + 1];
        const int64_t kblocks = kp / kSplitBK;
        const int64_t b = (int64_t)blockIdx.x - a_blocks;
        const int64_t k0 = (b % kblocks) * kSplitBK;
        const int64_t n0 = (b / kblocks) * kSplitBN;
        // read: 32 rows x 32 float4, four per thread, a warp per row
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int f = threadIdx.x + 256 * i;
            const int r = f >> 5, c = (f & 31) * 4;
            const int64_t k = k0 + r, n = n0 + c;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (k < K) {
                const float* src = B + k * ldb + n;
                if (vec_b && n + 3 < N) {
                    const float4 t = __ldg(reinterpret_cast<const float4*>(src));
                    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = (n + j < N) ? __ldg(src + j) : 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) tile[r][c + j] = v[j];
        }
        __syncthreads();
        // write: warp w takes columns n = 16w .. 16w+15, lane = k
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll 4
        for (int c = w * 16; c < w * 16 + 16; ++c) {
            const int64_t n = n0 + c;
            if (n < N) {
                float h, l;
                split3(tile[lane][c], h, l);
                b_hi[n * kp + k0 + lane] = h;
                b_lo[n * kp + k0 + lane] = l;
            }
        }
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Main kernel.
// ---------------------------------------------------------------------------

template <int BN, int STAGES>
struct TcLayout {
    static constexpr int A_BYTES = kBM * kBK * 4;   // 16 KB
    static constexpr int B_BYTES = BN * kBK * 4;
    static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    // cluster K-slice reduction: the receive buffer laid over the idle ring
    static constexpr bool CLUSTER_OK = ClusterSum<BN>::BYTES <= RING_BYTES;
    static constexpr bool FIXUP_OK = kFixRingBytes <= RING_BYTES;
    // full, empty, tmem x4, drain, full_b, ready, recv, stg, sumd, fixup loads x4
    static constexpr int NBARS = 3 * STAGES + 13;
    static constexpr int BAR_BYTES = 8 * NBARS + 16;
    // At least 116 KB, so that two CTAs never share an SM (each holds up to
    // all 512 TMEM columns for its whole lifetime).
    static constexpr int SMEM_USED = 1024 + RING_BYTES + BAR_BYTES;
    static constexpr int SMEM_BYTES = SMEM_USED > 116 * 1024 ? SMEM_USED : 116 * 1024;
    static constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulator buffers
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS >= 32 && TMEM_COLS <= 512, "TMEM cols");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// SEP = true is the ablation of the pages' barrier coalescing: the A and B
// tiles of a stage land on two separate "full" barriers (two expect-tx, two
// waits) instead of one.
template <int BN, int STAGES, bool SEP>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_ahi, const __grid_constant__ CUtensorMap tm_alo,
               const __grid_constant__ CUtensorMap tm_bhi, const __grid_constant__ CUtensorMap tm_blo,
               const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_p,
               const TcArgs args)
{
    using L = TcLayout<BN, STAGES>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Align the ring to 1024 B (128-byte swizzle atoms).
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t ring = (raw_addr + 1023u) & ~1023u;
    uint8_t* ring_ptr = smem_raw + (ring - raw_addr);
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring_ptr + L::RING_BYTES);
    // bars[0..S-1] full (A and B, or A only when SEP), [S..2S-1] empty,
    // [2S..2S+1] tmem_full, [2S+2..2S+3] tmem_empty, [2S+4] drain,
    // [2S+5..3S+4] full_b (SEP), [3S+5] ready, [3S+6] recv (cluster reduction);
    // then the TMEM base address slot and the abort flag.
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto full_bar = [&](int s) { return ptx::smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return ptx::smem_u32(bars + STAGES + s); };
    auto tfull_bar = [&](int b) { return ptx::smem_u32(bars + 2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return ptx::smem_u32(bars + 2 * STAGES + 2 + b); };
    const uint32_t drain_bar = ptx::smem_u32(bars + 2 * STAGES + 4);
    auto fullb_bar = [&](int s) { return ptx::smem_u32(bars + (SEP ? 2 * STAGES + 5 + s : s)); };
    const uint32_t ready_bar = ptx::smem_u32(bars + 3 * STAGES + 5);
    const uint32_t recv_bar = ptx::smem_u32(bars + 3 * STAGES + 6);
    const uint32_t stg_bar = ptx::smem_u32(bars + 3 * STAGES + 7);
    const uint32_t sum_bar = ptx::smem_u32(bars + 3 * STAGES + 8);
    auto fix_bar = [&](int q) { return ptx::smem_u32(bars + 3 * STAGES + 9 + q); };
    const bool clustered = L::CLUSTER_OK && args.cluster > 1;
    const bool fixup = L::FIXUP_OK && args.fixup && !clustered;

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
        if (SEP)
            for (int s = 0; s < STAGES; ++s) ptx::mbar_init(fullb_bar(s), 1);
        ptx::mbar_init(ready_bar, clustered ? args.cluster : 1);
        ptx::mbar_init(recv_bar, 1);
        ptx::mbar_init(stg_bar, 4);
        ptx::mbar_init(sum_bar, 4);
        for (int q = 0; q < 4; ++q) ptx::mbar_init(fix_bar(q), 1);
        // the S-1 incoming slices of this CTA's rows complete the one phase
        if (clustered)
            ptx::mbar_arrive_expect_tx(recv_bar, (uint32_t)((args.cluster - 1) *
                                                            ClusterSum<BN>::block_bytes(args.cluster)));
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
    // the peers' barriers are initialised before any remote arrival
    if (clustered) ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Programmatic launch: this grid may start while the previous kernel on the
    // stream (the split pre-pass, or the last GEMM) still runs.  Only the
    // producer reads global memory first, so only it waits for that kernel
    // (below); every other global access comes after its loads through the
    // mbarrier chain.  The next kernel may start its own prologue now.
    pdl_trigger();

    const int num_work = args.dp_tiles + args.split_tiles * args.splits;
    const int64_t limit = args.timeout;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            pdl_wait();  // the previous kernel's writes (split operands, C) are done
            int stage = 0;
            uint32_t phase = 0;
            uint32_t fills = 0;
            bool stop = false;
            for (int w = blockIdx.x; w < num_work && !stop; w += gridDim.x) {
                const Unit u = decode_unit(w, args);
                int tm, tn;
                tile_coords(u.tile, args.tiles_m, args.tiles_n, args.group, tm, tn);
                for (int kb = u.kb0; kb < u.kb1; ++kb) {
                    if (!wait_phase(empty_bar(stage), phase ^ 1u, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
                    ++fills;
                    if (fills != (uint32_t)args.withhold) {
                        const uint32_t sb = ring + stage * L::STAGE_BYTES;
                        const int kc = kb * kBK;
                        // One expect-tx covers all four operand tiles (A and B
                        // publish together); SEP arms A and B separately.
                        ptx::mbar_arrive_expect_tx(full_bar(stage), SEP ? 2 * L::A_BYTES : L::STAGE_BYTES);
                        ptx::tma_load_2d(sb, &tm_ahi, full_bar(stage), kc, tm * kBM);
                        ptx::tma_load_2d(sb + L::A_BYTES, &tm_alo, full_bar(stage), kc, tm * kBM);
                        if (SEP) ptx::mbar_arrive_expect_tx(fullb_bar(stage), 2 * L::B_BYTES);
                        ptx::tma_load_2d(sb + 2 * L::A_BYTES, &tm_bhi, fullb_bar(stage), kc, tn * BN);
                        ptx::tma_load_2d(sb + 2 * L::A_BYTES + L::B_BYTES, &tm_blo, fullb_bar(stage), kc,
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
                if (SEP) {
                    const long long t1 = clock64();
                    while (!ptx::mbar_try_wait(fullb_bar(s), par)) {
                        if (clock64() - t1 > limit) { atomicExch(args.status, kStatusTimeout); break; }
                    }
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
                const Unit u = decode_unit(w, args);
                const int kb0 = u.kb0, kb1 = u.kb1;
                const int buf = iter & 1;
                const uint32_t tphase = (iter >> 1) & 1;
                if (!wait_phase(tempty_bar(buf), tphase ^ 1u, limit, abort_flag, args.status)) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(full_bar(stage), phase, limit, abort_flag, args.status) ||
                        (SEP && !wait_phase(fullb_bar(stage), phase, limit, abort_flag, args.status))) {
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
        int iter = 0;
        for (int w = blockIdx.x; w < num_work; w += gridDim.x, ++iter) {
            const Unit u = decode_unit(w, args);
            int tm, tn;
            tile_coords(u.tile, args.tiles_m, args.tiles_n, args.group, tm, tn);
            const int buf = iter & 1;
            const uint32_t tphase = (iter >> 1) & 1;
            if (!wait_phase(tfull_bar(buf), tphase, limit, abort_flag, args.status)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + buf * BN;
            const EpilogueBars eb{ready_bar, recv_bar, stg_bar, sum_bar, fix_bar(quad)};
            if (!drain_unit<BN, L::RING_BYTES>(args, &tm_c, &tm_p, u, tm, tn, taddr, quad, lane,
                                               w + (int)gridDim.x >= num_work, clustered, fixup, ring, ring_ptr, eb,
                                               limit, abort_flag))
                break;
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty_bar(buf));
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    // no CTA of the cluster leaves while a peer may still reach its shared memory
    if (clustered) ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

// Sum the K-slices of every split tile in slice order and write the tile to C
// (guarded).  Grid-stride over split_tiles x 128 x BN/4 float4 positions.
template <int BN>
__global__ void __launch_bounds__(kReduceThreads, kReduceBlocksPerSm)
tile_reduce_kernel(const float4* __restrict__ partial, int dp_tiles, int split_tiles, int splits,
                   int tiles_m, int tiles_n, int group, int64_t M, int64_t N, float* __restrict__ C, int64_t ldc)
{
    pdl_trigger();  // the next kernel may start its prologue; it waits for this one itself
    pdl_wait();
    constexpr int Q = BN / 4;                 // float4 per partial row
    constexpr int PER_TILE = kBM * Q;
    const bool vec = ((ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(C) & 15) == 0);
    const int64_t total = (int64_t)split_tiles * PER_TILE;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(idx / PER_TILE);
        const int rem = (int)(idx % PER_TILE);
        const int r = rem / Q, c = (rem % Q) * 4;
        int tm, tn;
        tile_coords(dp_tiles + j, tiles_m, tiles_n, group, tm, tn);
        const int64_t grow = (int64_t)tm * kBM + r, gcol = (int64_t)tn * BN + c;
        if (grow >= M || gcol >= N) continue;
        const float4* p = partial + ((int64_t)j * splits * kBM + r) * Q + c / 4;
        const float4 acc = sum_slices<PER_TILE>(p, splits);
        float* dst = C + grow * ldc + gcol;
        if (vec && gcol + 3 < N) {
            *reinterpret_cast<float4*>(dst) = acc;
        } else {
            const float v[4] = {acc.x, acc.y, acc.z, acc.w};
            for (int q = 0; q < 4 && gcol + q < N; ++q) dst[q] = v[q];
        }
    }
}

}  // namespace
}  // namespace gemm_f32
