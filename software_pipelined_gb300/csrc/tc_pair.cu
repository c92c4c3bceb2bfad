// tcgen05 3xTF32 GEMM on CTA pairs: one 256 x BN output tile per pair of CTAs
// (a thread-block cluster of two), one tcgen05.mma.cta_group::2 for the pair.
//
// The same software pipeline as tc_fused.cu ("Double Buffering" technique page
// and "Case Study: The Double-Buffered GEMM": the next K-tile is fetched while
// the current one is multiplied), with the operand split inside the kernel,
// but the pair shares the work of staging the operands:
//
//   * each CTA holds its own 128 rows of A (raw by TMA, lo_A by its converter
//     warps) and HALF of the tile's B columns (raw 32 x 32 boxes by TMA,
//     transposed to hi_B / lo_B by its converters);
//   * or, in two lighter forms, B arrives split and transposed by the operand
//     pre-pass (hi_B and lo_B by TMA), and in the second of them lo_A too (hi
//     of A is the raw A, which the MMA truncates): then both CTAs' copies of
//     a stage complete on the even CTA's barrier (the TMA's cta_group::2 form
//     may signal the peer's barrier), and nothing sits between a stage's
//     copies and its MMAs;
//   * the even CTA's MMA thread issues M = 256, N = BN MMAs that read A rows
//     0..127 and B columns 0..BN/2-1 from its own shared memory and the rest
//     from its peer's, at the same addresses, and accumulate the even CTA's
//     128 rows in its TMEM and the odd CTA's 128 rows in the odd CTA's TMEM.
//
// Per CTA and k-block this halves the B tile a CTA copies, converts and feeds
// to the tensor core, against a 128 x BN tile of the one-CTA kernel with the
// same MMA work per SM, so the ring holds more stages.
//
// Synchronisation (every wait bounded; a CTA that gives up raises its own and
// its peer's abort flag):
//   full_a[s]  TMA of the CTA's raw A and B landed (local); in the form with
//              nothing to convert, the even CTA's barrier counts both CTAs'
//              copies (armed by the even CTA with the pair's bytes)
//   rd[s]      every converter warp (of the group on that stage) holds its
//              raw B (local)
//   conv[s]    (even CTA) both CTAs' converters are done: counts 2 x 4 warps
//              (one group of each CTA), the odd CTA's arriving remotely with
//              release at cluster scope (unused in the form with nothing to
//              convert)
//   empty[s]   the pair's MMAs of slot s completed: one commit, multicast to
//              both CTAs
//   tfull      accumulator complete: commit multicast to both CTAs
//   tempty     (even CTA) both CTAs' epilogues drained the accumulator: 8 warps
// Both CTAs take the same units in the same order.  Before they read any
// peer state they pass a cluster barrier, and before either exits (or frees
// TMEM) a second one, so no CTA leaves while its shared memory may still be
// read by the pair's MMAs or written by its peer.
#include <cstdint>

#include "tc_common.cuh"

namespace gemm_f32 {
namespace {

using namespace tc;
constexpr int kPairConvWarps = 8;
constexpr int kConvGroups = 2;                      // converter groups, on alternate stages
constexpr int kPairConvThreads = kPairConvWarps * 32;
constexpr int kPairThreads = 6 * 32 + kPairConvThreads;

// Where the pair kernel's operands are split.
enum : int {
    kPairSplitBoth = 0,  // raw A and raw B by TMA, both split by the converters
    kPairPreB = 1,       // hi_B, lo_B from the pre-pass; lo_A by the converters
    kPairPreAB = 2       // lo_A, hi_B, lo_B from the pre-pass; hi_A = raw A
};

// BN: the pair's tile width (each CTA holds BN/2 columns of B); KB: k per stage.
template <int BN, int SLOTS, int KB>
struct PairLayout {
    static constexpr int BH = BN / 2;                    // B columns per CTA
    static constexpr int A_BYTES = kBM * KB * 4;
    static constexpr int B_BYTES = BH * KB * 4;          // also raw B: BH/32 boxes
    static constexpr int BOX_BYTES = 32 * KB * 4;
    static_assert(KB == 32 || KB == 16, "stage depth");
    static_assert(BH % 32 == 0 && B_BYTES == BH / 32 * BOX_BYTES, "raw B fills the lo_B part exactly");
    static constexpr int SLOT_BYTES = 2 * A_BYTES + 2 * B_BYTES;
    static constexpr int RING_BYTES = SLOTS * SLOT_BYTES;
    // full, rd, conv, empty per slot + tfull/tempty x2, drain, ready, recv, spare
    static constexpr int NBARS = 4 * SLOTS + 8;
    static constexpr int BAR_BYTES = 8 * NBARS + 16;
    // B_BYTES of slack after the barriers: every MMA operand read of the pair
    // stays inside this CTA's allocation even if one ran BH rows past a slot
    static constexpr int SMEM_BYTES = 1024 + RING_BYTES + BAR_BYTES + B_BYTES;
    // Two accumulators of BN columns: a unit's epilogue drains one while the
    // next unit's MMAs fill the other.
    static constexpr int TBUFS = 2;
    static constexpr uint32_t TMEM_COLS = TBUFS * BN;
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM cols");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(RING_BYTES >= 4 * 8192, "the ring holds the TMA-store staging");
};

template <int KB>
__device__ __forceinline__ uint32_t pair_kmajor_off(int row, int kq)
{
    if constexpr (KB == 32)
        return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((kq ^ (row & 7)) << 4));
    else
        return (uint32_t)((row >> 3) * 512 + (row & 7) * 64 + ((kq ^ ((row >> 1) & 3)) << 4));
}

template <int KB>
__device__ __forceinline__ uint64_t pair_kmajor_desc(uint32_t saddr)
{
    if constexpr (KB == 32) {
        return sw128_desc(saddr);
    } else {
        return (uint64_t)((saddr & 0x3FFFFu) >> 4)
             | ((uint64_t)1 << 16)                  // leading byte offset (unused)
             | ((uint64_t)(512 >> 4) << 32)         // stride byte offset: 8 rows of 64 B
             | ((uint64_t)1 << 46)                  // descriptor version (tcgen05)
             | ((uint64_t)4 << 61);                 // swizzle: 64 B
    }
}

// Instruction descriptor, kind::tf32, M = 256 (a CTA pair), N = BN.
template <int BN>
__host__ __device__ constexpr uint32_t idesc_tf32_pair()
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}

// The unit of a pair in pair tiles (dp_tiles, split_tiles in pair tiles), and
// this CTA's 128-row tile and partial slot in it.  Pair tile P covers tile
// rows 2*ptm and 2*ptm + 1 of tile column tn, (ptm, tn) in the grouped order
// over pair rows; a split pair tile q's slice z goes to slots
// (2q + rank) * splits + z, so that tile j = 2q + rank of the split tiles
// owns slots j * splits .. j * splits + splits - 1.
struct PairUnit {
    Unit u;      // this CTA's share: tile = 2P + rank, kb range, slot (-1: C)
    int tm, tn;  // this CTA's 128-row tile
};

__device__ __forceinline__ PairUnit pair_unit(int w, const TcArgs& a, int rank)
{
    const Unit pu = decode_unit(w, a);
    PairUnit r;
    int ptm, tn;
    tile_coords(pu.tile, a.tiles_m / 2, a.tiles_n, a.group, ptm, tn);
    r.tm = 2 * ptm + rank;
    r.tn = tn;
    r.u.tile = 2 * pu.tile + rank;
    r.u.kb0 = pu.kb0;
    r.u.kb1 = pu.kb1;
    if (pu.slot < 0) {
        r.u.slot = -1;
    } else {
        const int q = pu.slot / a.splits, z = pu.slot % a.splits;
        r.u.slot = (2 * q + rank) * a.splits + z;
    }
    return r;
}

// The K-slice sum of a tile inside a cluster of S pairs (S = 2 or 4; the pairs
// are the tile's S K-slices, slice z = cluster rank / 2).  The S CTAs holding
// the same 128-row half h of the tile form a group; in it, slice z owns
// quadrants (32-row blocks) z*4/S .. (z+1)*4/S - 1 and sums them.  Per
// epilogue warp (quadrant q of this CTA's accumulator), once the accumulator
// is complete (the ring is idle):
//   * one thread tells every group member that this ring is free (`ready`,
//     S arrivals);
//   * a warp whose quadrant another slice owns stages it in the ring (32 x 32
//     swizzled boxes) and, once every group member is ready, pushes it with
//     one bulk copy into the owner's receive slot for this slice, completing
//     on the owner's `recv` barrier (armed at start for all incoming bytes);
//   * a warp of an owned quadrant waits for `recv`, adds the S slices in slice
//     order (this slice's from TMEM; the order of the reduction kernel, so the
//     same bits) and stores C.
// Ring layout: the 4 - 4/S quadrants staged out, then (S-1) x 4/S received
// blocks.  Every wait bounded; false means this warp gave up.
template <int BN>
struct PairSum {
    static constexpr int QUAD_BYTES = 32 * BN * 4;
    static constexpr __host__ __device__ int ring_bytes(int S) { return (4 - 4 / S + (S - 1) * (4 / S)) * QUAD_BYTES; }
};

template <int BN>
__device__ bool pair_cluster_sum(const TcArgs& args, const CUtensorMap* tm_c, int tm, int tn, uint32_t taddr,
                                 int quad, int lane, int z, int h, uint32_t ring, uint8_t* ring_ptr,
                                 uint32_t ready_bar, uint32_t recv_bar, int64_t limit, volatile int* abort_flag)
{
    constexpr int QB = PairSum<BN>::QUAD_BYTES, NB = BN / 32;
    const int S = args.cluster, qpo = 4 / S, own0 = z * qpo;
    const int owner = quad / qpo;
    const uint32_t recv = ring + (4 - qpo) * QB;
    uint8_t* recv_ptr = ring_ptr + (4 - qpo) * QB;
    if (quad == 0 && lane == 0)
        for (int g = 0; g < S; ++g) ptx::mbar_arrive_cluster(ptx::mapa(ready_bar, (uint32_t)(2 * g + h)));
    if (owner != z) {
        const int slot = quad < own0 ? quad : quad - qpo;  // staging slot of this quadrant
        uint8_t* stg_ptr = ring_ptr + slot * QB;
#pragma unroll 1
        for (int bx = 0; bx < NB; ++bx) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x16(taddr + bx * 32, *reinterpret_cast<uint32_t(*)[16]>(r));
            ptx::tmem_ld_32x32b_x16(taddr + bx * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
            ptx::tmem_wait_ld();
            stage_row(stg_ptr + bx * 4096, lane, r);
        }
        ptx::fence_proxy_async_shared();  // generic-proxy writes -> the bulk copy's reads
        __syncwarp();
        int ok = 1;
        if (lane == 0) {
            ok = wait_phase_cluster(ready_bar, 0, limit, abort_flag, args.status);
            if (ok) {
                const int rs = (z < owner ? z : z - 1) * qpo + (quad - owner * qpo);  // owner's receive slot
                const uint32_t dst = (uint32_t)(2 * owner + h);
                ptx::bulk_copy_to_cluster(ptx::mapa(recv + rs * QB, dst), ring + slot * QB, (uint32_t)QB,
                                          ptx::mapa(recv_bar, dst));
            }
        }
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    }
    if (!__all_sync(0xffffffffu, wait_phase_cluster(recv_bar, 0, limit, abort_flag, args.status))) return false;
    const int i = quad - own0;
    const int64_t grow = (int64_t)tm * kBM + quad * 32 + lane;
    const bool vec = ((args.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(args.C) & 15) == 0);
#pragma unroll 1
    for (int bx = 0; bx < NB; ++bx) {
        float acc[32];
#pragma unroll 1
        for (int sl = 0; sl < S; ++sl) {
            if (sl == z) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t r[16];
                    ptx::tmem_ld_32x32b_x16(taddr + bx * 32 + hh * 16, r);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        acc[hh * 16 + c] = sl == 0 ? __uint_as_float(r[c]) : acc[hh * 16 + c] + __uint_as_float(r[c]);
                }
            } else {
                const uint8_t* row = recv_ptr + ((sl < z ? sl : sl - 1) * qpo + i) * QB + bx * 4096 + lane * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 t = *reinterpret_cast<const float4*>(row + ((q ^ (lane & 7)) << 4));
                    if (sl == 0) {
                        acc[4 * q] = t.x; acc[4 * q + 1] = t.y; acc[4 * q + 2] = t.z; acc[4 * q + 3] = t.w;
                    } else {
                        acc[4 * q] += t.x; acc[4 * q + 1] += t.y; acc[4 * q + 2] += t.z; acc[4 * q + 3] += t.w;
                    }
                }
            }
        }
        const int64_t gcol = (int64_t)tn * BN + bx * 32;
        if (grow < args.M && gcol < args.N) {
            float* dst = args.C + grow * args.ldc + gcol;
            if (vec && gcol + 31 < args.N) {
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    *reinterpret_cast<float4*>(dst + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (gcol + c < args.N) dst[c] = acc[c];
            }
        }
    }
    return true;
}

// The split pair tiles' K-slices summed in slice order into C, float4 by
// float4: indices idx0, idx0 + step, ... of 2 x split_pairs dense 128 x BN
// partial tiles (slice z of the half h of split pair tile q at slot
// (2q + h) x splits + z).  COHERENT: the slices were written by other CTAs of
// the running kernel (loads through L2 only).
template <int BN, bool COHERENT>
__device__ __forceinline__ void pair_reduce_range(const float4* __restrict__ partial, int dp_pairs, int split_pairs,
                                                  int splits, int tiles_m, int tiles_n, int group, int64_t M,
                                                  int64_t N, float* __restrict__ C, int64_t ldc, int64_t idx0,
                                                  int64_t step)
{
    constexpr int Q = BN / 4;
    constexpr int PER_TILE = kBM * Q;
    const bool vec = ((ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(C) & 15) == 0);
    const int64_t total = (int64_t)2 * split_pairs * PER_TILE;
    for (int64_t idx = idx0; idx < total; idx += step) {
        const int j = (int)(idx / PER_TILE);
        const int rem = (int)(idx % PER_TILE);
        const int r = rem / Q, c = (rem % Q) * 4;
        int ptm, tn;
        tile_coords(dp_pairs + j / 2, tiles_m / 2, tiles_n, group, ptm, tn);
        const int64_t grow = ((int64_t)2 * ptm + (j & 1)) * kBM + r, gcol = (int64_t)tn * BN + c;
        if (grow >= M || gcol >= N) continue;
        const float4* p = partial + ((int64_t)j * splits * kBM + r) * Q + c / 4;
        const float4 acc = sum_slices<PER_TILE, COHERENT>(p, splits);
        float* dst = C + grow * ldc + gcol;
        if (vec && gcol + 3 < N) {
            *reinterpret_cast<float4*>(dst) = acc;
        } else {
            const float v[4] = {acc.x, acc.y, acc.z, acc.w};
            for (int q = 0; q < 4 && gcol + q < N; ++q) dst[q] = v[q];
        }
    }
}

// The grid sum of a pair kernel, out of line so that its registers do not
// weigh on the kernel's main loop: the grid-wide barrier, then this CTA's
// share of the slices' sums.
template <int BN>
__device__ __noinline__ void pair_grid_sum(const TcArgs& args, volatile int* ok_word)
{
    ptx::fence_proxy_async_global();
    if (grid_barrier(reinterpret_cast<unsigned*>(args.sem), args.timeout, args.status, ok_word))
        pair_reduce_range<BN, true>(reinterpret_cast<const float4*>(args.partial), args.dp_tiles, args.split_tiles,
                                    args.splits, args.tiles_m, args.tiles_n, args.group, args.M, args.N, args.C,
                                    args.ldc, (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
                                    (int64_t)gridDim.x * blockDim.x);
}

// MODE kPairPreB: B comes split and transposed by the pre-pass (hi and lo,
// K-major, by TMA through tm_bhi / tm_blo: this CTA's half of the tile's
// columns) and the converters only add lo_A; kPairPreAB: lo_A comes from the
// pre-pass as well (tm_alo) and the converters convert nothing;
// kPairSplitBoth: tm_b copies raw B boxes and the converters split both
// operands.  The pre-split operands' tensor maps have boxes of KB k.
template <int BN, int SLOTS, int KB, int MODE>
__global__ void __launch_bounds__(kPairThreads, 1)
tc_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_bhi, const __grid_constant__ CUtensorMap tm_blo,
               const __grid_constant__ CUtensorMap tm_alo, const __grid_constant__ CUtensorMap tm_c,
               const __grid_constant__ CUtensorMap tm_p, const TcArgs args)
{
    constexpr bool BPRE = MODE != kPairSplitBoth;
    constexpr bool APRE = MODE == kPairPreAB;
    static_assert(MODE != kPairPreB || KB == 32, "the hybrid form runs 32-k stages");
    using L = PairLayout<BN, SLOTS, KB>;
    constexpr int HALVES = kBK / KB;  // stages per 32-k block of the work decomposition
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t ring = (raw_addr + 1023u) & ~1023u;
    uint8_t* ring_ptr = smem_raw + (ring - raw_addr);
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring_ptr + L::RING_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The cluster is one pair, or (the K-slice sum in distributed shared
    // memory) the S pairs of a tile's S K-slices: cluster rank = 2 x slice + rank
    // in the pair.  The pair's even CTA issues its MMAs.
    const uint32_t crank = ptx::cluster_ctarank();
    const uint32_t rank = crank & 1u, lead = crank & ~1u;
    const uint16_t pair_mask = (uint16_t)(3u << lead);
    const bool clustered = args.cluster > 1;
    auto full_a = [&](int s) { return ptx::smem_u32(bars + s); };
    auto conv = [&](int s) { return ptx::smem_u32(bars + SLOTS + s); };
    auto empty = [&](int s) { return ptx::smem_u32(bars + 2 * SLOTS + s); };
    auto rd = [&](int s) { return ptx::smem_u32(bars + 3 * SLOTS + s); };
    auto tfull = [&](int b) { return ptx::smem_u32(bars + 4 * SLOTS + b); };
    auto tempty = [&](int b) { return ptx::smem_u32(bars + 4 * SLOTS + 2 + b); };
    const uint32_t drain_bar = ptx::smem_u32(bars + 4 * SLOTS + 4);
    const uint32_t ready_bar = ptx::smem_u32(bars + 4 * SLOTS + 5);  // cluster sum: the group's rings are idle
    const uint32_t recv_bar = ptx::smem_u32(bars + 4 * SLOTS + 6);   // cluster sum: the owned blocks landed
    // the abort flag of the peer CTA (shared::cluster address)
    const uint32_t peer_abort = ptx::mapa(ptx::smem_u32(const_cast<int*>(abort_flag)), crank ^ 1u);
    auto give_up = [&]() {
        *abort_flag = 1;
        ptx::st_cluster_u32(peer_abort, 1u);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < SLOTS; ++s) {
            ptx::mbar_init(full_a(s), 1);
            // one group of each CTA's converters
            ptx::mbar_init(conv(s), 2 * kPairConvWarps / kConvGroups);
            ptx::mbar_init(empty(s), 1);
            ptx::mbar_init(rd(s), kPairConvWarps / kConvGroups);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull(b), 1);
            ptx::mbar_init(tempty(b), 8);
        }
        ptx::mbar_init(drain_bar, 1);
        ptx::mbar_init(ready_bar, clustered ? args.cluster : 1);
        ptx::mbar_init(recv_bar, 1);
        // the S-1 other slices' blocks of this CTA's owned quadrants complete the one phase
        if (clustered)
            ptx::mbar_arrive_expect_tx(recv_bar, (uint32_t)((args.cluster - 1) * PairSum<BN>::QUAD_BYTES * 4 /
                                                            args.cluster));
        *abort_flag = 0;
        ptx::mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tm_a);
        if (APRE) ptx::tma_prefetch_desc(&tm_alo);
        if (BPRE) {
            ptx::tma_prefetch_desc(&tm_bhi);
            ptx::tma_prefetch_desc(&tm_blo);
        } else {
            ptx::tma_prefetch_desc(&tm_b);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), L::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    // both CTAs' barriers initialised, TMEM allocated, abort flags cleared
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_trigger();

    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int num_work = args.dp_tiles + args.split_tiles * args.splits;
    const int64_t limit = args.timeout;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            pdl_wait();  // the previous kernel's writes (A, B, C) are done
            uint32_t fills = 0;
            bool stop = false;
            for (int w = pair; w < num_work && !stop; w += npairs) {
                const PairUnit pu = pair_unit(w, args, (int)rank);
                for (int kh = pu.u.kb0 * HALVES; kh < pu.u.kb1 * HALVES; ++kh) {
                    const int s = fills % SLOTS;
                    const uint32_t ps = (fills / SLOTS) & 1u;
                    if (!wait_phase(empty(s), ps ^ 1u, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
                    ++fills;
                    if (fills == (uint32_t)args.withhold) continue;
                    const int kc = kh * KB;
                    const uint32_t slot = ring + s * L::SLOT_BYTES;
                    if constexpr (APRE) {
                        // raw A (= hi_A) and lo_A, this CTA's half of hi_B and lo_B;
                        // both CTAs' copies complete on the even CTA's barrier, which
                        // the even CTA's thread arms with the pair's bytes
                        if (rank == 0) ptx::mbar_arrive_expect_tx(full_a(s), 2 * (2 * L::A_BYTES + 2 * L::B_BYTES));
                        const uint32_t fb = rank == 0 ? full_a(s) : ptx::mapa(full_a(s), lead);
                        ptx::tma_load_2d_pair(slot, &tm_a, fb, kc, pu.tm * kBM);
                        ptx::tma_load_2d_pair(slot + L::A_BYTES, &tm_alo, fb, kc, pu.tm * kBM);
                        const int n0 = pu.tn * BN + (int)rank * L::BH;
                        ptx::tma_load_2d_pair(slot + 2 * L::A_BYTES, &tm_bhi, fb, kc, n0);
                        ptx::tma_load_2d_pair(slot + 2 * L::A_BYTES + L::B_BYTES, &tm_blo, fb, kc, n0);
                    } else if constexpr (BPRE) {
                        // raw A into the A part, this CTA's half of hi_B and lo_B
                        ptx::mbar_arrive_expect_tx(full_a(s), L::A_BYTES + 2 * L::B_BYTES);
                        ptx::tma_load_2d(slot, &tm_a, full_a(s), kc, pu.tm * kBM);
                        const int n0 = pu.tn * BN + (int)rank * L::BH;
                        ptx::tma_load_2d(slot + 2 * L::A_BYTES, &tm_bhi, full_a(s), kc, n0);
                        ptx::tma_load_2d(slot + 2 * L::A_BYTES + L::B_BYTES, &tm_blo, full_a(s), kc, n0);
                    } else {
                        // raw A (this CTA's 128 rows) into the A part, raw B boxes
                        // (this CTA's half of the columns) into the lo_B part
                        ptx::mbar_arrive_expect_tx(full_a(s), L::A_BYTES + L::B_BYTES);
                        ptx::tma_load_2d(slot, &tm_a, full_a(s), kc, pu.tm * kBM);
#pragma unroll
                        for (int j = 0; j < L::BH / 32; ++j)
                            ptx::tma_load_2d(slot + 2 * L::A_BYTES + L::B_BYTES + j * L::BOX_BYTES, &tm_b,
                                             full_a(s), pu.tn * BN + (int)rank * L::BH + 32 * j, kc);
                    }
                }
            }
            if (stop) give_up();
            // Drain: the last fill of every slot must have landed.  With every
            // piece by TMA the odd CTA's copies complete on the even CTA's
            // barriers, so the even CTA's drain covers both CTAs (and the odd
            // CTA leaves only after it, at the final cluster barrier); after
            // an abort the odd CTA gives a copy it issued without a matching
            // copy of the even CTA time to land.
            const uint32_t total = fills;
            if (APRE && rank == 1) {
                if (stop) {
                    const long long t0 = clock64();
                    while (clock64() - t0 < (1 << 20)) {
                    }
                }
            } else {
                for (int s = 0; s < SLOTS && (uint32_t)s < total; ++s) {
                    const uint32_t last = (total - 1 - s) / SLOTS * SLOTS + s;
                    if (last + 1 == (uint32_t)args.withhold) continue;
                    const uint32_t par = (last / SLOTS) & 1u;
                    const long long t0 = clock64();
                    while (!ptx::mbar_try_wait(full_a(s), par))
                        if (clock64() - t0 > limit) { atomicExch(args.status, kStatusTimeout); break; }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_tf32_pair<BN>();
            uint32_t fills = 0;
            int iter = 0;
            bool stop = false;
            for (int w = pair; w < num_work && !stop; w += npairs, ++iter) {
                const Unit u = decode_unit(w, args);
                const int buf = L::TBUFS == 2 ? (iter & 1) : 0;
                const uint32_t tphase = (uint32_t)(iter / L::TBUFS) & 1u;
                if (!wait_phase_cluster(tempty(buf), tphase ^ 1u, limit, abort_flag, args.status)) {
                    stop = true;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kh = u.kb0 * HALVES; kh < u.kb1 * HALVES; ++kh, ++fills) {
                    const int s = fills % SLOTS;
                    const uint32_t ps = (fills / SLOTS) & 1u;
                    if (APRE ? !wait_phase(full_a(s), ps, limit, abort_flag, args.status)
                             : !wait_phase_cluster(conv(s), ps, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_hi = ring + s * L::SLOT_BYTES, a_lo = a_hi + L::A_BYTES;
                    const uint32_t b_hi = a_hi + 2 * L::A_BYTES, b_lo = b_hi + L::B_BYTES;
#pragma unroll
                    for (int ks = 0; ks < KB / kUmmaK; ++ks) {
                        const uint32_t off = ks * kUmmaK * 4;
                        const uint32_t acc = (kh > u.kb0 * HALVES || ks > 0) ? 1u : 0u;
                        if (args.terms == 3) {
                            ptx::mma_tf32_pair(d_tmem, pair_kmajor_desc<KB>(a_lo + off),
                                               pair_kmajor_desc<KB>(b_hi + off), idesc, acc);
                            ptx::mma_tf32_pair(d_tmem, pair_kmajor_desc<KB>(a_hi + off),
                                               pair_kmajor_desc<KB>(b_lo + off), idesc, 1u);
                            ptx::mma_tf32_pair(d_tmem, pair_kmajor_desc<KB>(a_hi + off),
                                               pair_kmajor_desc<KB>(b_hi + off), idesc, 1u);
                        } else {
                            ptx::mma_tf32_pair(d_tmem, pair_kmajor_desc<KB>(a_hi + off),
                                               pair_kmajor_desc<KB>(b_hi + off), idesc, acc);
                        }
                    }
                    ptx::mma_commit_pair(empty(s), pair_mask);  // both CTAs' slot s free once these finish
                }
                if (stop) break;
                ptx::mma_commit_pair(tfull(buf), pair_mask);  // both CTAs' accumulators complete
            }
            if (stop) give_up();
            ptx::mma_commit_pair(drain_bar, (uint16_t)(1u << lead));
            const long long t0 = clock64();
            while (!ptx::mbar_try_wait(drain_bar, 0))
                if (clock64() - t0 > limit) { atomicExch(args.status, kStatusTimeout); break; }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------ epilogue ------------------------------
        const int quad = warp & 3;
        const uint32_t lead_tempty0 = ptx::mapa(tempty(0), lead), lead_tempty1 = ptx::mapa(tempty(1), lead);
        int iter = 0;
        bool stop = false;
        for (int w = pair; w < num_work; w += npairs, ++iter) {
            const PairUnit pu = pair_unit(w, args, (int)rank);
            const int buf = L::TBUFS == 2 ? (iter & 1) : 0;
            const uint32_t tphase = (uint32_t)(iter / L::TBUFS) & 1u;
            if (!wait_phase(tfull(buf), tphase, limit, abort_flag, args.status)) {
                stop = true;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + buf * BN;
            if (clustered) {
                if (!pair_cluster_sum<BN>(args, &tm_c, pu.tm, pu.tn, taddr, quad, lane, (int)(crank >> 1),
                                          (int)rank, ring, ring_ptr, ready_bar, recv_bar, limit, abort_flag)) {
                    stop = true;
                    break;
                }
            } else {
                const EpilogueBars eb{drain_bar, drain_bar, drain_bar, drain_bar, drain_bar};  // unused
                drain_unit<BN, L::RING_BYTES>(args, &tm_c, &tm_p, pu.u, pu.tm, pu.tn, taddr, quad, lane,
                                              w + npairs >= num_work, false, false, ring, ring_ptr, eb, limit,
                                              abort_flag);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(buf ? lead_tempty1 : lead_tempty0);
        }
        if (stop && lane == 0) give_up();
    } else if constexpr (APRE) {
        // nothing to convert: the converter warps idle
    } else {
        // ------------------------------ converters ----------------------------
        // Two groups of warps take alternate stages, so that one group's
        // per-stage synchronisation (the raw-B hand-over, the proxy fence, the
        // release to the even CTA) overlaps the other group's conversion.
        constexpr int GW = kPairConvWarps / kConvGroups;  // warps per group
        constexpr int KG = KB / 4;                         // 4-wide k groups per stage
        constexpr int NBOX = L::BH / 32;                   // raw-B boxes per stage
        constexpr int PER = KG * NBOX / GW;                // (k group, box) pairs per warp
        static_assert(PER >= 1 && PER * GW == KG * NBOX, "converter work split");
        const int ct = threadIdx.x - 6 * 32;  // 0 .. kPairConvThreads-1
        const int grp = (ct >> 5) / GW, gw = (ct >> 5) % GW;
        const int gt = ct - grp * GW * 32;    // thread index in the group
        uint32_t fills = 0;
        bool stop = false;
        for (int w = pair; w < num_work && !stop; w += npairs) {
            const Unit u = decode_unit(w, args);
            for (int kh = u.kb0 * HALVES; kh < u.kb1 * HALVES; ++kh, ++fills) {
                if ((int)(fills % kConvGroups) != grp) continue;  // the other group's stage
                const int s = fills % SLOTS;
                const uint32_t ps = (fills / SLOTS) & 1u;
                // The slot's previous use may belong to the other group, and its
                // copy may land after this group's last one: wait until the MMAs
                // released it, so that the parity wait below is for this use.
                if (fills >= (uint32_t)SLOTS && !wait_phase(empty(s), ps ^ 1u, limit, abort_flag, args.status)) {
                    stop = true;
                    break;
                }
                if (!wait_phase(full_a(s), ps, limit, abort_flag, args.status)) {
                    stop = true;
                    break;
                }
                uint8_t* slot = ring_ptr + s * L::SLOT_BYTES;
                const uint8_t* a_raw = slot;
                uint8_t* a_lo = slot + L::A_BYTES;
                uint8_t* b_hi = slot + 2 * L::A_BYTES;
                uint8_t* b_lo = b_hi + L::B_BYTES;  // holds raw B until every warp of the group has read it
                // B: this warp's (k group, box) pairs into registers (row k of a
                // box: chunk (lane/4) ^ (k%8), word lane%4), hi_B written at once.
                float v[PER][4];
                if constexpr (!BPRE) {
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    const int pr = gw + i * GW, cw = pr % KG, nb = pr / KG;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int k = cw * 4 + j;
                        v[i][j] = *reinterpret_cast<const float*>(
                            b_lo + nb * L::BOX_BYTES + k * 128 + (((lane >> 2) ^ (k & 7)) << 4) + (lane & 3) * 4);
                    }
                    *reinterpret_cast<float4*>(b_hi + pair_kmajor_off<KB>(nb * 32 + lane, cw)) =
                        make_float4(v[i][0], v[i][1], v[i][2], v[i][3]);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(rd(s));
                }
#pragma unroll
                for (int c = gt; c < L::A_BYTES / 16; c += GW * 32) {
                    const float4 x = *reinterpret_cast<const float4*>(a_raw + c * 16);
                    *reinterpret_cast<float4*>(a_lo + c * 16) =
                        make_float4(lo_part(x.x), lo_part(x.y), lo_part(x.z), lo_part(x.w));
                }
                if constexpr (!BPRE) {
                    if (!wait_phase(rd(s), ps, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
#pragma unroll
                    for (int i = 0; i < PER; ++i) {
                        const int pr = gw + i * GW, cw = pr % KG, nb = pr / KG;
                        *reinterpret_cast<float4*>(b_lo + pair_kmajor_off<KB>(nb * 32 + lane, cw)) =
                            make_float4(lo_part(v[i][0]), lo_part(v[i][1]), lo_part(v[i][2]), lo_part(v[i][3]));
                    }
                }
                ptx::fence_proxy_async_shared();  // generic-proxy writes -> the pair's tensor-core reads
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(conv(s), lead));
            }
        }
        if (stop && lane == 0) give_up();
    }

    ptx::tc_fence_before();
    __syncthreads();
    // no CTA leaves (or frees TMEM) while the pair's MMAs may still read its
    // shared memory or its peer may still arrive on its barriers
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
    }
    // Every unit of the grid stored (the epilogues waited for their bulk
    // stores): the split tiles' slices summed by the whole grid, in the
    // reduction kernel's order.  The idle ring holds the barrier's word.
    if (args.gridsum) pair_grid_sum<BN>(args, reinterpret_cast<volatile int*>(ring_ptr));
}

// ---------------------------------------------------------------------------
// CTA pairs with A in tensor memory.
//
// The pair tile is 256 x 256 as above, but A's pieces never sit in shared
// memory while the MMAs run: raw A comes by TMA into a small staging ring
// (16 KB a stage), four loader warps of each CTA (one thread per row of the
// CTA's 128 rows) read their rows from it, split them in registers (hi = the
// value truncated to TF32, lo = the remainder rounded to TF32), free the
// staging slot, and write both pieces into a ring of A slots in tensor memory
// with tcgen05.st; the MMAs take A from there (the tcgen05.mma form whose A
// operand is in tensor memory, each CTA of the pair providing its 128 rows).
// Shared memory then holds this CTA's half of hi_B and lo_B (split and
// transposed by the pre-pass) 5 stages deep and raw A 3 stages deep, where
// the 64 KB stages of the forms above fit 3 in all, and no pre-pass writes or
// reads lo of A.  Tensor memory (512 columns): one 256-column accumulator (a
// unit's epilogue drains it before the next unit's MMAs start) and 4 A slots
// of 64 columns (hi in the first 32, lo in the next).
//
// Barriers (every wait bounded; a CTA that gives up raises both abort flags):
//   s_full[j]   raw A of staging slot j landed (TMA, local)
//   s_empty[j]  this CTA's 4 loader warps have read staging slot j (local)
//   b_full[s]   (even CTA) both CTAs' hi_B / lo_B halves of stage s landed
//               (TMA; the odd CTA's copies signal it directly)
//   b_empty[s]  the pair's MMAs of B slot s completed (commit, multicast)
//   a_full[t]   (even CTA) both CTAs' loader warps wrote A slot t: 8 arrivals
//   a_empty[t]  the pair's MMAs of A slot t completed (commit, multicast)
//   tfull       the accumulator is complete (commit, multicast)
//   tempty      (even CTA) both CTAs' epilogues drained it: 8 arrivals
template <int NB_SLOTS, int NA_STAGE>
struct TmemALayout {
    static constexpr int BN = 256, BH = 128, KB = 32;
    static constexpr int A_SLOTS = 4;
    static constexpr int B_BYTES = BH * KB * 4;     // one piece of this CTA's half of B
    static constexpr int SLOT_BYTES = 2 * B_BYTES;  // hi_B, lo_B
    static constexpr int RING_BYTES = NB_SLOTS * SLOT_BYTES;
    static constexpr int STAGE_A_BYTES = kBM * KB * 4;  // raw A of one stage: 128 rows x 32
    static constexpr int NBARS = 2 * NB_SLOTS + 2 * A_SLOTS + 2 * NA_STAGE + 3;
    static constexpr int BAR_BYTES = 8 * NBARS + 16;
    // B_BYTES of slack after the barriers, as in PairLayout
    static constexpr int SMEM_BYTES = 1024 + RING_BYTES + NA_STAGE * STAGE_A_BYTES + BAR_BYTES + B_BYTES;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t A_COL0 = 256;         // A slot t: columns A_COL0 + 64 t (hi), + 32 (lo)
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(RING_BYTES >= 4 * 8 * 4096, "the ring holds the last unit's TMA-store staging");
};
// B producer, MMA, 4 epilogue, 4 loader warps, A producer
constexpr int kTmemAThreads = 11 * 32;

template <int NB_SLOTS, int NA_STAGE>
__global__ void __launch_bounds__(kTmemAThreads, 1)
tc_pair_tmem_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_bhi,
                    const __grid_constant__ CUtensorMap tm_blo, const __grid_constant__ CUtensorMap tm_c,
                    const __grid_constant__ CUtensorMap tm_p, const TcArgs args)
{
    using L = TmemALayout<NB_SLOTS, NA_STAGE>;
    constexpr int BN = L::BN, SA = L::A_SLOTS, SB = NB_SLOTS, SS = NA_STAGE;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t ring = (raw_addr + 1023u) & ~1023u;
    uint8_t* ring_ptr = smem_raw + (ring - raw_addr);
    const uint32_t astage = ring + L::RING_BYTES;  // raw A staging, after the B ring
    const uint8_t* astage_ptr = ring_ptr + L::RING_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring_ptr + L::RING_BYTES + SS * L::STAGE_A_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = ptx::cluster_ctarank();
    const uint32_t rank = crank & 1u, lead = crank & ~1u;
    const uint16_t pair_mask = (uint16_t)(3u << lead);
    auto b_full = [&](int s) { return ptx::smem_u32(bars + s); };
    auto b_empty = [&](int s) { return ptx::smem_u32(bars + SB + s); };
    auto a_full = [&](int t) { return ptx::smem_u32(bars + 2 * SB + t); };
    auto a_empty = [&](int t) { return ptx::smem_u32(bars + 2 * SB + SA + t); };
    const uint32_t tfull = ptx::smem_u32(bars + 2 * SB + 2 * SA);
    const uint32_t tempty = ptx::smem_u32(bars + 2 * SB + 2 * SA + 1);
    const uint32_t drain_bar = ptx::smem_u32(bars + 2 * SB + 2 * SA + 2);
    auto s_full = [&](int j) { return ptx::smem_u32(bars + 2 * SB + 2 * SA + 3 + j); };
    auto s_empty = [&](int j) { return ptx::smem_u32(bars + 2 * SB + 2 * SA + 3 + SS + j); };
    const uint32_t peer_abort = ptx::mapa(ptx::smem_u32(const_cast<int*>(abort_flag)), crank ^ 1u);
    auto give_up = [&]() {
        *abort_flag = 1;
        ptx::st_cluster_u32(peer_abort, 1u);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < SB; ++s) {
            ptx::mbar_init(b_full(s), 1);
            ptx::mbar_init(b_empty(s), 1);
        }
        for (int t = 0; t < SA; ++t) {
            ptx::mbar_init(a_full(t), 8);
            ptx::mbar_init(a_empty(t), 1);
        }
        ptx::mbar_init(tfull, 1);
        ptx::mbar_init(tempty, 8);
        ptx::mbar_init(drain_bar, 1);
        for (int j = 0; j < SS; ++j) {
            ptx::mbar_init(s_full(j), 1);
            ptx::mbar_init(s_empty(j), 4);
        }
        *abort_flag = 0;
        ptx::mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tm_a);
        ptx::tma_prefetch_desc(&tm_bhi);
        ptx::tma_prefetch_desc(&tm_blo);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), L::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    // both CTAs' barriers initialised, TMEM allocated, abort flags cleared
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_trigger();

    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int num_work = args.dp_tiles + args.split_tiles * args.splits;
    const int64_t limit = args.timeout;

    if (warp == 0) {
        // ----------------------------- B producer -----------------------------
        if (lane == 0) {
            pdl_wait();  // the previous kernel's writes (split B, C) are done
            uint32_t fills = 0;
            bool stop = false;
            for (int w = pair; w < num_work && !stop; w += npairs) {
                const PairUnit pu = pair_unit(w, args, (int)rank);
                for (int kb = pu.u.kb0; kb < pu.u.kb1; ++kb) {
                    const int s = fills % SB;
                    const uint32_t ps = (fills / SB) & 1u;
                    if (!wait_phase(b_empty(s), ps ^ 1u, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
                    ++fills;
                    if (fills == (uint32_t)args.withhold) continue;
                    const uint32_t slot = ring + s * L::SLOT_BYTES;
                    const int n0 = pu.tn * BN + (int)rank * L::BH;
                    // both CTAs' halves complete on the even CTA's barrier
                    if (rank == 0) ptx::mbar_arrive_expect_tx(b_full(s), 2 * L::SLOT_BYTES);
                    const uint32_t fb = rank == 0 ? b_full(s) : ptx::mapa(b_full(s), lead);
                    ptx::tma_load_2d_pair(slot, &tm_bhi, fb, kb * L::KB, n0);
                    ptx::tma_load_2d_pair(slot + L::B_BYTES, &tm_blo, fb, kb * L::KB, n0);
                }
            }
            if (stop) give_up();
            // Drain: the last fill of every slot must have landed (the even
            // CTA's barriers count both CTAs' copies; after an abort the odd
            // CTA gives a copy without a matching copy of the even CTA time to
            // land).
            const uint32_t total = fills;
            if (rank == 1) {
                if (stop) {
                    const long long t0 = clock64();
                    while (clock64() - t0 < (1 << 20)) {
                    }
                }
            } else {
                for (int s = 0; s < SB && (uint32_t)s < total; ++s) {
                    const uint32_t last = (total - 1 - s) / SB * SB + s;
                    if (last + 1 == (uint32_t)args.withhold) continue;
                    const uint32_t par = (last / SB) & 1u;
                    const long long t0 = clock64();
                    while (!ptx::mbar_try_wait(b_full(s), par))
                        if (clock64() - t0 > limit) { atomicExch(args.status, kStatusTimeout); break; }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_tf32_pair<BN>();
            uint32_t fills = 0;
            int iter = 0;
            bool stop = false;
            for (int w = pair; w < num_work && !stop; w += npairs, ++iter) {
                const Unit u = decode_unit(w, args);
                // the single accumulator: the last unit's epilogues drained it
                if (!wait_phase_cluster(tempty, ((uint32_t)iter & 1u) ^ 1u, limit, abort_flag, args.status)) {
                    stop = true;
                    break;
                }
                ptx::tc_fence_after();
                for (int kb = u.kb0; kb < u.kb1; ++kb, ++fills) {
                    const int s = fills % SB, t = fills % SA;
                    const uint32_t ps = (fills / SB) & 1u, pt = (fills / SA) & 1u;
                    if (!wait_phase(b_full(s), ps, limit, abort_flag, args.status) ||
                        !wait_phase_cluster(a_full(t), pt, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t b_hi = ring + s * L::SLOT_BYTES, b_lo = b_hi + L::B_BYTES;
                    const uint32_t a_hi = tmem_base + L::A_COL0 + (uint32_t)t * 64u, a_lo = a_hi + 32u;
#pragma unroll
                    for (int ks = 0; ks < L::KB / kUmmaK; ++ks) {
                        const uint32_t boff = ks * kUmmaK * 4, acol = ks * kUmmaK;
                        const uint32_t acc = (kb > u.kb0 || ks > 0) ? 1u : 0u;
                        if (args.terms == 3) {
                            ptx::mma_tf32_pair_ts(tmem_base, a_lo + acol, sw128_desc(b_hi + boff), idesc, acc);
                            ptx::mma_tf32_pair_ts(tmem_base, a_hi + acol, sw128_desc(b_lo + boff), idesc, 1u);
                            ptx::mma_tf32_pair_ts(tmem_base, a_hi + acol, sw128_desc(b_hi + boff), idesc, 1u);
                        } else {
                            ptx::mma_tf32_pair_ts(tmem_base, a_hi + acol, sw128_desc(b_hi + boff), idesc, acc);
                        }
                    }
                    // both CTAs' B slot s and A slot t are free once these finish
                    ptx::mma_commit_pair(b_empty(s), pair_mask);
                    ptx::mma_commit_pair(a_empty(t), pair_mask);
                }
                if (stop) break;
                ptx::mma_commit_pair(tfull, pair_mask);  // both CTAs' accumulators complete
            }
            if (stop) give_up();
            ptx::mma_commit_pair(drain_bar, (uint16_t)(1u << lead));
            const long long t0 = clock64();
            while (!ptx::mbar_try_wait(drain_bar, 0))
                if (clock64() - t0 > limit) { atomicExch(args.status, kStatusTimeout); break; }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------ epilogue ------------------------------
        const int quad = warp & 3;
        const uint32_t lead_tempty = ptx::mapa(tempty, lead);
        int iter = 0;
        bool stop = false;
        for (int w = pair; w < num_work; w += npairs, ++iter) {
            const PairUnit pu = pair_unit(w, args, (int)rank);
            if (!wait_phase(tfull, (uint32_t)iter & 1u, limit, abort_flag, args.status)) {
                stop = true;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16);
            const EpilogueBars eb{drain_bar, drain_bar, drain_bar, drain_bar, drain_bar};  // unused
            drain_unit<BN, L::RING_BYTES>(args, &tm_c, &tm_p, pu.u, pu.tm, pu.tn, taddr, quad, lane,
                                          w + npairs >= num_work, false, false, ring, ring_ptr, eb, limit,
                                          abort_flag);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(lead_tempty);
        }
        if (stop && lane == 0) give_up();
    } else if (warp < 10) {
        // ------------------------------ A loaders -----------------------------
        // Warp w owns TMEM lanes 32 (w % 4) .. +31, i.e. those rows of this
        // CTA's 128; a lane is one row.  Per 32-k block: the row's 128 bytes
        // from the staging slot (16-byte chunks in the 128-byte swizzle, so a
        // quarter-warp's 8 rows hit 8 distinct bank groups), the slot handed
        // back, hi and lo written to A slot t, the slot handed to the even CTA
        // (8 arrivals: 4 warps of each CTA).
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        uint32_t fills = 0;
        bool stop = false;
        for (int w = pair; w < num_work && !stop; w += npairs) {
            const Unit u = decode_unit(w, args);
            for (int kb = u.kb0; kb < u.kb1; ++kb, ++fills) {
                const int j = fills % SS, t = fills % SA;
                const uint32_t pj = (fills / SS) & 1u, pt = (fills / SA) & 1u;
                if (!__all_sync(0xffffffffu, wait_phase(s_full(j), pj, limit, abort_flag, args.status))) {
                    stop = true;
                    break;
                }
                const uint8_t* src = astage_ptr + j * L::STAGE_A_BYTES + row * 128;
                float v[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 q = *reinterpret_cast<const float4*>(src + ((c ^ (row & 7)) << 4));
                    v[4 * c] = q.x; v[4 * c + 1] = q.y; v[4 * c + 2] = q.z; v[4 * c + 3] = q.w;
                }
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    hi[c] = __float_as_uint(v[c]) & 0xFFFFE000u;  // what the MMA reads of the raw value
                    lo[c] = __float_as_uint(lo_part(v[c]));
                }
                // these generic-proxy reads before the TMA's next write of the slot
                ptx::fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(s_empty(j));
                // the MMAs of this slot's last use are done
                if (!__all_sync(0xffffffffu, wait_phase(a_empty(t), pt ^ 1u, limit, abort_flag, args.status))) {
                    stop = true;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t slot = tmem_base + lane_off + L::A_COL0 + (uint32_t)t * 64u;
                ptx::tmem_st_32x32b_x32(slot, hi);
                ptx::tmem_st_32x32b_x32(slot + 32u, lo);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(a_full(t), lead));
            }
        }
        if (stop && lane == 0) give_up();
    } else {
        // ----------------------------- A producer -----------------------------
        // Raw A of this CTA's 128 rows, one 32-k block per staging slot, in
        // the loaders' order; rows past M and k past K read as zero.
        if (lane == 0) {
            pdl_wait();  // the previous kernel's writes (A) are done
            uint32_t fills = 0;
            bool stop = false;
            for (int w = pair; w < num_work && !stop; w += npairs) {
                const PairUnit pu = pair_unit(w, args, (int)rank);
                for (int kb = pu.u.kb0; kb < pu.u.kb1; ++kb) {
                    const int j = fills % SS;
                    const uint32_t pj = (fills / SS) & 1u;
                    if (!wait_phase(s_empty(j), pj ^ 1u, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
                    ++fills;
                    ptx::mbar_arrive_expect_tx(s_full(j), L::STAGE_A_BYTES);
                    ptx::tma_load_2d(astage + j * L::STAGE_A_BYTES, &tm_a, s_full(j), kb * L::KB, pu.tm * kBM);
                }
            }
            if (stop) give_up();
            // Drain: the last fill of every slot must have landed.
            const uint32_t total = fills;
            for (int j = 0; j < SS && (uint32_t)j < total; ++j) {
                const uint32_t last = (total - 1 - j) / SS * SS + j;
                const uint32_t par = (last / SS) & 1u;
                const long long t0 = clock64();
                while (!ptx::mbar_try_wait(s_full(j), par))
                    if (clock64() - t0 > limit) { atomicExch(args.status, kStatusTimeout); break; }
            }
        }
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    // no CTA leaves (or frees TMEM) while the pair's MMAs may still read its
    // shared or tensor memory or its peer may still arrive on its barriers
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
    }
}

template <int NB, int NS>
cudaError_t launch_pair_tmem(const TcPlanState& st, const TcArgs& a, const CUtensorMap& ta,
                             const CUtensorMap& tbhi, const CUtensorMap& tblo, cudaStream_t s)
{
    using L = TmemALayout<NB, NS>;
    auto kern = tc_pair_tmem_kernel<NB, NS>;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = smem_limit_once(kern, L::SMEM_BYTES, smem_set); e != cudaSuccess) return e;
    const int work = a.dp_tiles + a.split_tiles * a.splits;
    const int pairs = work < st.pair_slots ? work : st.pair_slots;
    if (pairs < 1 || a.cluster > 1) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3(2 * pairs), dim3(kTmemAThreads), L::SMEM_BYTES, s, 2, ta, tbhi, tblo,
                      *reinterpret_cast<const CUtensorMap*>(st.tmap_c),
                      *reinterpret_cast<const CUtensorMap*>(st.tmap_p), a);
}

template <int NB, int NS>
int pair_tmem_slots_for(int sms)
{
    using L = TmemALayout<NB, NS>;
    auto kern = tc_pair_tmem_kernel<NB, NS>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2 > 0 ? sms / 2 : 1));
    cfg.blockDim = dim3(kTmemAThreads);
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// Sum the K-slices of every split pair tile (its two 128-row tiles) in slice
// order and write C (guarded).  Grid-stride over 2 x split_tiles (pairs) x 128
// x BN/4 float4 positions; tile j = 2q + r of the split tiles is row half r of
// split pair tile q.
template <int BN>
__global__ void __launch_bounds__(kReduceThreads, kReduceBlocksPerSm)
pair_reduce_kernel(const float4* __restrict__ partial, int dp_pairs, int split_pairs, int splits, int tiles_m,
                   int tiles_n, int group, int64_t M, int64_t N, float* __restrict__ C, int64_t ldc)
{
    pdl_trigger();
    pdl_wait();
    pair_reduce_range<BN, false>(partial, dp_pairs, split_pairs, splits, tiles_m, tiles_n, group, M, N, C, ldc,
                                 (int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
}

template <int BN, int SLOTS, int KB, int MODE>
cudaError_t launch_pair(const TcPlanState& st, const TcArgs& a, const CUtensorMap& ta, const CUtensorMap& tb,
                        const CUtensorMap& tbhi, const CUtensorMap& tblo, const CUtensorMap& talo, cudaStream_t s)
{
    using L = PairLayout<BN, SLOTS, KB>;
    auto kern = tc_pair_kernel<BN, SLOTS, KB, MODE>;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = smem_limit_once(kern, L::SMEM_BYTES, smem_set); e != cudaSuccess) return e;
    const int work = a.dp_tiles + a.split_tiles * a.splits;
    // cluster sum: every pair its one unit, the S pairs of a tile one cluster
    const int pairs = a.cluster > 1 ? work : (work < st.pair_slots ? work : st.pair_slots);
    if (pairs < 1) return cudaErrorInvalidValue;
    if (a.cluster > 1 && (a.dp_tiles != 0 || a.splits != a.cluster ||
                          PairSum<BN>::ring_bytes(a.cluster) > L::RING_BYTES))
        return cudaErrorInvalidValue;
    // the grid sum's barrier needs every CTA resident at once
    return launch_pdl_ex(kern, dim3(2 * pairs), dim3(kPairThreads), L::SMEM_BYTES, s,
                         a.cluster > 1 ? 2 * a.cluster : 2, a.gridsum != 0, ta, tb, tbhi, tblo, talo,
                         *reinterpret_cast<const CUtensorMap*>(st.tmap_c),
                         *reinterpret_cast<const CUtensorMap*>(st.tmap_p), a);
}

template <int BN, int SLOTS, int KB>
int pair_slots_for(int sms)
{
    using L = PairLayout<BN, SLOTS, KB>;
    auto kern = tc_pair_kernel<BN, SLOTS, KB, kPairSplitBoth>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2 > 0 ? sms / 2 : 1));
    cfg.blockDim = dim3(kPairThreads);
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace

cudaError_t tc_pair_main(int bn, int bk, int split, const TcPlanState& st, const TcArgs& a,
                         const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbhi,
                         const CUtensorMap& tblo, const CUtensorMap& talo, cudaStream_t s)
{
    if (split == kSplitRawA) {
        if (bn == 256 && bk == 32) return launch_pair<256, 3, 32, kPairPreAB>(st, a, ta, tb, tbhi, tblo, talo, s);
        if (bn == 256 && bk == 16) return launch_pair<256, 6, 16, kPairPreAB>(st, a, ta, tb, tbhi, tblo, talo, s);
        if (bn == 128 && bk == 32) return launch_pair<128, 4, 32, kPairPreAB>(st, a, ta, tb, tbhi, tblo, talo, s);
        return cudaErrorInvalidValue;
    }
    if (split == kSplitHybrid) {
        if (bn == 256 && bk == 32) return launch_pair<256, 3, 32, kPairPreB>(st, a, ta, tb, tbhi, tblo, talo, s);
        if (bn == 128 && bk == 32) return launch_pair<128, 4, 32, kPairPreB>(st, a, ta, tb, tbhi, tblo, talo, s);
        return cudaErrorInvalidValue;
    }
    if (split != kSplitInKernel) return cudaErrorInvalidValue;
    if (bn == 256 && bk == 32) return launch_pair<256, 3, 32, kPairSplitBoth>(st, a, ta, tb, tbhi, tblo, talo, s);
    if (bn == 256 && bk == 16) return launch_pair<256, 6, 16, kPairSplitBoth>(st, a, ta, tb, tbhi, tblo, talo, s);
    if (bn == 128 && bk == 32) return launch_pair<128, 4, 32, kPairSplitBoth>(st, a, ta, tb, tbhi, tblo, talo, s);
    if (bn == 128 && bk == 16) return launch_pair<128, 8, 16, kPairSplitBoth>(st, a, ta, tb, tbhi, tblo, talo, s);
    return cudaErrorInvalidValue;
}

cudaError_t tc_pair_tmem_main(const TcPlanState& st, const TcArgs& a, const CUtensorMap& ta,
                              const CUtensorMap& tbhi, const CUtensorMap& tblo, cudaStream_t s)
{
    return launch_pair_tmem<5, 3>(st, a, ta, tbhi, tblo, s);
}

cudaError_t tc_pair_reduce(int bn, const TcPlanState& st, const TcArgs& a, cudaStream_t s)
{
    const int64_t total = (int64_t)2 * a.split_tiles * kBM * (bn / 4);
    const dim3 grid(reduce_blocks(total, st.num_sms));
    const float4* p = reinterpret_cast<const float4*>(a.partial);
    if (bn == 256)
        return launch_pdl(pair_reduce_kernel<256>, grid, dim3(kReduceThreads), 0, s, 1, p, a.dp_tiles, a.split_tiles, a.splits,
                          a.tiles_m, a.tiles_n, a.group, a.M, a.N, a.C, a.ldc);
    if (bn == 128)
        return launch_pdl(pair_reduce_kernel<128>, grid, dim3(kReduceThreads), 0, s, 1, p, a.dp_tiles, a.split_tiles, a.splits,
                          a.tiles_m, a.tiles_n, a.group, a.M, a.N, a.C, a.ldc);
    return cudaErrorInvalidValue;
}

int tc_pair_slots(int bn, int bk, int sms, int split)
{
    if (split == kSplitTmemA) return bn == 256 && bk == 32 ? pair_tmem_slots_for<5, 3>(sms) : 0;
    // the same shared memory and threads for every other form of the operands
    if (bn == 256 && bk == 32) return pair_slots_for<256, 3, 32>(sms);
    if (bn == 256 && bk == 16) return pair_slots_for<256, 6, 16>(sms);
    if (bn == 128 && bk == 32) return pair_slots_for<128, 4, 32>(sms);
    if (bn == 128 && bk == 16) return pair_slots_for<128, 8, 16>(sms);
    return 0;
}

}  // namespace gemm_f32
