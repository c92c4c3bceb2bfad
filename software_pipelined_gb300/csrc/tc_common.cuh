// Device helpers shared by the two tensor-core GEMM kernels (operands split
// by a pre-pass, in tc_gemm.cu; split inside the kernel, in tc_fused.cu):
// the unit-of-work decomposition, tcgen05 descriptors, bounded mbarrier waits,
// the tile order, the TMEM epilogue and launches with programmatic stream
// serialisation.
#pragma once
#include <cstdint>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gemm_f32 {
namespace tc {

constexpr int kBM = 128;      // tile rows = TMEM lanes
constexpr int kBK = 32;       // fp32 elements per 128-byte swizzle row
constexpr int kUmmaK = 8;     // K of one kind::tf32 MMA
constexpr int64_t kDefaultTimeout = int64_t(1) << 32;  // SM clock cycles

struct TcArgs {
    int64_t M, N;
    int64_t ldc;
    float* C;
    float* partial;      // split units' dense 128 x BN partial tiles
    int* status;
    int64_t timeout;
    int tiles_m, tiles_n;
    int num_kb;          // k-blocks of 32 in the padded K
    int dp_tiles;        // tiles computed whole, written to C
    int split_tiles;     // tiles computed in `splits` K-slices each
    int splits;
    int kb_per_split;
    int terms;           // 3 = 3xTF32, 1 = hi*hi only
    int withhold;        // test hook: 1-based fill index the producer skips (0 = none)
    int group;           // tile-rows per raster group of the tile order
    int c_tma;           // 1: the C tensor map is valid (C 16-byte aligned, ldc % 4 == 0)
    int* sem;            // fixup: one arrival counter per (split tile, 32-row quadrant), or NULL
    int fixup;           // 1: split units sum their tile's slices themselves (last arriver)
    int cluster;         // > 1: every tile split in `cluster` K-slices, one CTA each, the
                         // slices of a tile one thread-block cluster that sums them
                         // through distributed shared memory (no partial tiles)
    int gridsum;         // 1: CTA pairs, cooperative grid: once every CTA has stored its
                         // units, a grid-wide barrier (sem[0] count, sem[1] generation),
                         // then every CTA sums a share of the split tiles' slices
};

// One unit of work of the persistent kernel: a whole tile, or one K-slice of a
// split tile.
struct Unit {
    int tile;            // index in tile order
    int kb0, kb1;        // k-block range
    int slot;            // -1: write C; else index of the dense partial tile
};

__device__ __forceinline__ Unit decode_unit(int w, const TcArgs& a)
{
    Unit u;
    if (w < a.dp_tiles) {
        u.tile = w;
        u.kb0 = 0;
        u.kb1 = a.num_kb;
        u.slot = -1;
    } else {
        const int t = w - a.dp_tiles;
        const int z = t % a.splits;
        u.tile = a.dp_tiles + t / a.splits;
        u.kb0 = z * a.kb_per_split;
        u.kb1 = min(a.num_kb, u.kb0 + a.kb_per_split);
        u.slot = t;
    }
    return u;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Round an FP32 value to the nearest TF32 value (10 explicit mantissa bits),
// ties to even, by integer arithmetic on the bit pattern; the low 13 bits of
// the result are zero.  Inf stays Inf; NaN stays NaN.  A finite x whose
// rounding would carry into the Inf exponent (|x| >= 0x7F7FF000, the top 4096
// FP32 values) is truncated instead: there |x| is within 2^-11 of 2^128, so
// one TF32 ulp (2^117) is at most 2^-11 |x| and x - hi stays as small,
// relative to x, as a rounded remainder anywhere else.  So no finite x gives
// a non-finite piece.
__device__ __forceinline__ float tf32_rne(float x)
{
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7F800000u) != 0x7F800000u) {
        const uint32_t r = u + 0x0FFFu + ((u >> 13) & 1u);
        if ((r & 0x7F800000u) != 0x7F800000u) u = r;
    }
    return __uint_as_float(u & 0xFFFFE000u);
}

__device__ __forceinline__ void split3(float x, float& hi, float& lo)
{
    hi = tf32_rne(x);
    lo = tf32_rne(x - hi);  // x - hi is exact in FP32
}

// Truncate an FP32 value to TF32 (the low 13 bits cleared): what a kind::tf32
// MMA makes of an FP32 operand.
__device__ __forceinline__ float tf32_trunc(float x)
{
    return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// lo = RN(x - trunc_tf32(x)) to 11 significant bits, ties away from zero: the
// difference is exact in FP32; adding half an ulp of TF32 to the magnitude and
// clearing the low 13 bits rounds it.  Two integer and one float operation per
// element (plus the truncation), no special cases: for finite x the result is
// finite; a non-finite x makes the hi*hi product non-finite anyway.
__device__ __forceinline__ float lo_part(float x)
{
    const float d = x - tf32_trunc(x);
    return __uint_as_float((__float_as_uint(d) + 0x1000u) & 0xFFFFE000u);
}

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

// The same bounded wait on a barrier that other CTAs of the cluster arrive on
// (acquire at cluster scope).
__device__ __forceinline__ bool wait_phase_cluster(uint32_t bar, uint32_t parity, int64_t limit,
                                                   volatile int* abort_flag, int* status)
{
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            atomicExch(status, kStatusTimeout);
            *abort_flag = 1;
            return false;
        }
    }
}

// Tile order: groups of G tile-rows, column-major inside a group, so the CTAs
// running together share A and B panels in L2.
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int G, int& tm, int& tn)
{
    const int group_size = G * tiles_n;
    const int gid = tile / group_size;
    const int first_m = gid * G;
    const int gsz = min(tiles_m - first_m, G);
    const int r = tile % group_size;
    tm = first_m + r % gsz;
    tn = r / gsz;
}

// Drain one accumulator buffer of TMEM (this warp's 32 lanes = 32 tile rows)
// into C (whole tiles, guarded, 16-byte stores where C allows) or into a dense
// 128 x BN partial tile (K-slices).
template <int BN>
__device__ __forceinline__ void store_accumulator(const TcArgs& args, const Unit& u, int tm, int tn,
                                                  uint32_t taddr, int row_in_tile)
{
    float* orow;
    int64_t col0, ncols;
    bool vec, row_ok;
    if (u.slot < 0) {
        const int64_t grow = (int64_t)tm * kBM + row_in_tile;
        row_ok = grow < args.M;
        orow = args.C + (row_ok ? grow : 0) * args.ldc;
        col0 = (int64_t)tn * BN;
        ncols = args.N;
        vec = ((args.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(args.C) & 15) == 0);
    } else {
        // all of the partial tile (rows past M hold the zero-filled operands' zeros)
        row_ok = true;
        orow = args.partial + ((int64_t)u.slot * kBM + row_in_tile) * BN;
        col0 = 0;
        ncols = BN;
        vec = true;
    }
#pragma unroll 1
    for (int c = 0; c < BN; c += 16) {
        uint32_t r[16];
        ptx::tmem_ld_32x32b_x16(taddr + c, r);
        ptx::tmem_wait_ld();
        const int64_t gn = col0 + c;
        if (row_ok) {
            if (vec && gn + 15 < ncols) {
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4*>(orow + gn + j) =
                        make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                    __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (gn + j < ncols) orow[gn + j] = __uint_as_float(r[j]);
            }
        }
    }
}

// Write 32 FP32 of one row (this lane) into a 32 x 32 box of the 128-byte
// swizzled layout (16-byte chunk q of row r at chunk q ^ (r % 8)): the 8 lanes
// of each store phase hit 8 different chunks, so no bank conflicts.
__device__ __forceinline__ void stage_row(uint8_t* box, int lane, const uint32_t* r)
{
    uint8_t* row = box + lane * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(row + ((q ^ (lane & 7)) << 4)) =
            make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
}

// Epilogue through TMA stores, for a CTA's last unit (its operand ring is then
// idle and serves as staging).  The calling warp owns TMEM lanes = tile rows
// y0 .. y0+31 of the destination (C, or the partial-tile buffer) and NBUF
// staging boxes of 32 rows x 32 FP32 (4 KB each) from `stage`.  Boxes go in
// pairs: four TMEM loads (64 columns) and one wait, two staged boxes, two TMA
// stores (clipped at the tensor's edge; boxes wholly past it are neither
// staged nor stored, so every staged box is one committed group).  A box
// buffer is reused only once the store that read it is done.
template <int BN, int NBUF>
__device__ __forceinline__ void store_accumulator_tma(const CUtensorMap* map, int64_t x0, int64_t y0,
                                                      int64_t xlim, int64_t ylim, uint32_t taddr, int lane,
                                                      uint32_t stage, uint8_t* stage_ptr)
{
    static_assert(NBUF >= 2 && BN % 64 == 0, "box pairs");
    const int cols = y0 < ylim ? (int)(xlim - x0 < BN ? xlim - x0 : BN) : 0;
    const int nbox = (cols + 31) >> 5;
#pragma unroll 1
    for (int j = 0; j < nbox; j += 2) {
        if (j + 1 >= NBUF) {
            // boxes up to j + 1 - NBUF (the previous users of these buffers) are read
            if (lane == 0) ptx::bulk_wait_read<NBUF - 2>();
            __syncwarp();
        }
        uint32_t r[64];
#pragma unroll
        for (int h = 0; h < 4; ++h)
            ptx::tmem_ld_32x32b_x16(taddr + j * 32 + h * 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16 * h));
        ptx::tmem_wait_ld();
        stage_row(stage_ptr + (j % NBUF) * 4096, lane, r);
        if (j + 1 < nbox) stage_row(stage_ptr + ((j + 1) % NBUF) * 4096, lane, r + 32);
        ptx::fence_proxy_async_shared();  // generic-proxy writes -> the TMA engine's reads
        __syncwarp();
        if (lane == 0) {
            ptx::tma_store_2d(map, stage + (j % NBUF) * 4096, (int32_t)(x0 + j * 32), (int32_t)y0);
            ptx::bulk_commit();
            if (j + 1 < nbox) {
                ptx::tma_store_2d(map, stage + ((j + 1) % NBUF) * 4096, (int32_t)(x0 + j * 32 + 32), (int32_t)y0);
                ptx::bulk_commit();
            }
        }
    }
    if (lane == 0) ptx::bulk_wait_all();  // complete before the staging is reused or freed
    __syncwarp();
}

// Last-arriver sum of a split tile's K-slices, for split units that are their
// CTA's last unit (the ring is idle and gives each epilogue warp kFixWarpBytes
// of staging).  Per warp, i.e. per 32-row quadrant of the tile:
//   1. this slice's rows of the partial tile go out by TMA and complete;
//   2. the warp counts its arrival on the (tile, quadrant) counter (proxy
//      fence and release before, so the rows are visible to whoever reads);
//   3. the warp that arrives S-th reads the other S-1 slices' rows box by box
//      (TMA loads), adds them to its own rows (TMEM) in slice order - the
//      reduction kernel's order, so the same bits - stores the sums to C and
//      resets the counter for the next run.
// No warp ever waits for another CTA; every wait is bounded.  false = a wait
// gave up (status set).
constexpr int kFixLoadBoxes = 7;                            // other slices: S <= 8
constexpr int kFixWarpBytes = (kFixLoadBoxes + 2) * 4096;   // + two output boxes
constexpr int kFixRingBytes = 4 * kFixWarpBytes;            // 144 KB of ring

template <int BN>
__device__ bool fixup_store(const TcArgs& args, const CUtensorMap* tm_p, const CUtensorMap* tm_c, const Unit& u,
                            int tm, int tn, uint32_t taddr, int quad, int lane, uint32_t stage, uint8_t* stage_ptr,
                            uint32_t ld_bar, int64_t limit, volatile int* abort_flag)
{
    constexpr int NB = BN / 32;
    constexpr int NSTORE = NB < kFixLoadBoxes + 2 ? NB : kFixLoadBoxes + 2;
    const int S = args.splits;
    const int j = u.slot / S, mine = u.slot % S;
    // 1.
    store_accumulator_tma<BN, NSTORE>(tm_p, 0, (int64_t)u.slot * kBM + quad * 32, BN, INT64_MAX, taddr, lane,
                                      stage, stage_ptr);
    // 2.
    int* counter = args.sem + j * 4 + quad;
    int old = 0;
    if (lane == 0) {
        ptx::fence_proxy_async_global();
        __threadfence();
        old = atomicAdd(counter, 1);
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != S - 1) return true;
    // 3. the last arriver
    if (lane == 0) {
        __threadfence();
        ptx::fence_proxy_async_global();
        *reinterpret_cast<volatile int*>(counter) = 0;
    }
    __syncwarp();
    const bool vec = ((args.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(args.C) & 15) == 0);
    const int64_t y = (int64_t)tm * kBM + quad * 32;
    // only the boxes that reach into C: each one is stored (one bulk group)
    const int64_t ncols = args.N - (int64_t)tn * BN;
    const int nb = y < args.M ? (int)((ncols < BN ? ncols : BN) + 31) / 32 : 0;
#pragma unroll 1
    for (int b = 0; b < nb; ++b) {
        const int64_t x = (int64_t)tn * BN + b * 32;
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(ld_bar, (uint32_t)((S - 1) * 4096));
            for (int z = 0, i = 0; z < S; ++z)
                if (z != mine)
                    ptx::tma_load_2d(stage + (i++) * 4096, tm_p, ld_bar, b * 32, (j * S + z) * kBM + quad * 32);
        }
        uint32_t own[32];
        ptx::tmem_ld_32x32b_x16(taddr + b * 32, *reinterpret_cast<uint32_t(*)[16]>(own));
        ptx::tmem_ld_32x32b_x16(taddr + b * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(own + 16));
        ptx::tmem_wait_ld();
        if (!__all_sync(0xffffffffu, wait_phase(ld_bar, (uint32_t)(b & 1), limit, abort_flag, args.status)))
            return false;
        uint32_t sum[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int off = lane * 128 + ((q ^ (lane & 7)) << 4);
            float4 acc;
            for (int z = 0, i = 0; z < S; ++z) {
                float4 v;
                if (z == mine) {
                    v = make_float4(__uint_as_float(own[4 * q]), __uint_as_float(own[4 * q + 1]),
                                    __uint_as_float(own[4 * q + 2]), __uint_as_float(own[4 * q + 3]));
                } else {
                    v = *reinterpret_cast<const float4*>(stage_ptr + (i++) * 4096 + off);
                }
                if (z == 0) {
                    acc = v;
                } else {
                    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
                }
            }
            sum[4 * q] = __float_as_uint(acc.x); sum[4 * q + 1] = __float_as_uint(acc.y);
            sum[4 * q + 2] = __float_as_uint(acc.z); sum[4 * q + 3] = __float_as_uint(acc.w);
        }
        ptx::fence_proxy_async_shared();  // these generic reads before the next box's TMA writes
        if (args.c_tma) {
            const int ob = kFixLoadBoxes + (b & 1);
            if (b >= 2) {
                if (lane == 0) ptx::bulk_wait_read<1>();  // output box ob stored two boxes ago
                __syncwarp();
            }
            stage_row(stage_ptr + ob * 4096, lane, sum);
            ptx::fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
                ptx::tma_store_2d(tm_c, stage + ob * 4096, (int32_t)x, (int32_t)y);
                ptx::bulk_commit();
            }
        } else {
            __syncwarp();
            const int64_t grow = y + lane;
            if (grow < args.M) {
                float* row = args.C + grow * args.ldc;
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const int64_t gcol = x + c;
                    if (vec && gcol + 3 < args.N) {
                        *reinterpret_cast<float4*>(row + gcol) =
                            make_float4(__uint_as_float(sum[c]), __uint_as_float(sum[c + 1]),
                                        __uint_as_float(sum[c + 2]), __uint_as_float(sum[c + 3]));
                    } else {
                        for (int k = 0; k < 4 && gcol + k < args.N; ++k) row[gcol + k] = __uint_as_float(sum[c + k]);
                    }
                }
            }
        }
    }
    if (lane == 0) ptx::bulk_wait_all();
    __syncwarp();
    return true;
}

// Shared-memory plan of the cluster K-slice sum, laid over the idle ring:
// STG holds this CTA's whole accumulator as 32 x 32 swizzled boxes, quadrant
// (32 rows) by quadrant; RECV holds the peers' slices of the rows this CTA
// owns, one slot per slice.  Rank r owns quadrants r*4/S .. (r+1)*4/S - 1, a
// contiguous block of STG, so each slice travels as one bulk copy.
template <int BN>
struct ClusterSum {
    static constexpr int QUAD_BYTES = 32 * BN * 4;
    static constexpr int STG_BYTES = 4 * QUAD_BYTES;
    static constexpr int BYTES = 2 * STG_BYTES;     // STG + RECV (S slots of a block)
    static __device__ __forceinline__ int block_bytes(int S) { return (4 / S) * QUAD_BYTES; }
};

// Epilogue of a K-sliced tile whose S = args.cluster (2 or 4) slices are the
// S CTAs of one cluster (rank z = slice z).  Called by the 128 epilogue
// threads (e = TMEM lane = tile row) once this CTA's accumulator is complete.
//   1. The ring is idle: one thread arrives on every rank's `ready` barrier.
//   2. Each warp stages its quadrant into STG; `stg` (4 arrivals) marks it.
//   3. One thread waits for `stg` and for `ready` (S arrivals: every ring is
//      free), then pushes the block of each owner p != z from STG into slot z
//      of p's RECV with one bulk copy that completes on p's `recv` barrier
//      (armed at start for the S-1 incoming blocks).
//   4. Everyone waits for `recv` (the S-1 blocks landed) and `stg`, sums the
//      S slices of the owned block in slice order (the reduction kernel's
//      order: the same bits) into STG, and marks it on `sumd` (4 arrivals).
//   5. The owned boxes go to C by TMA stores (or by direct stores when C
//      cannot take them).
// Every wait is bounded; false means one gave up (status set).  No CTA
// leaves before the cluster barrier at the kernel's end, so no remote access
// targets an exited CTA.
template <int BN>
__device__ bool cluster_reduce_store(const TcArgs& args, const CUtensorMap* tm_c, int tm, int tn,
                                     uint32_t taddr, int quad, int lane, uint32_t ring, uint8_t* ring_ptr,
                                     uint32_t ready_bar, uint32_t recv_bar, uint32_t stg_bar, uint32_t sum_bar,
                                     int64_t limit, volatile int* abort_flag)
{
    using CS = ClusterSum<BN>;
    constexpr int NB = BN / 32;  // boxes per quadrant row
    const int S = args.cluster;
    const int e = quad * 32 + lane;
    const uint32_t z = ptx::cluster_ctarank();
    const int block = CS::block_bytes(S);
    const uint32_t stg = ring, recv = ring + CS::STG_BYTES;
    uint8_t* stg_ptr = ring_ptr;
    const uint8_t* recv_ptr = ring_ptr + CS::STG_BYTES;
    // 1.
    if (e == 0)
        for (int r = 0; r < S; ++r) ptx::mbar_arrive_cluster(ptx::mapa(ready_bar, (uint32_t)r));
    // 2.
#pragma unroll 1
    for (int bx = 0; bx < NB; ++bx) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x16(taddr + bx * 32, *reinterpret_cast<uint32_t(*)[16]>(r));
        ptx::tmem_ld_32x32b_x16(taddr + bx * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
        ptx::tmem_wait_ld();
        stage_row(stg_ptr + (quad * NB + bx) * 4096, lane, r);
    }
    ptx::fence_proxy_async_shared();  // visible to the bulk copies that read STG
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(stg_bar);
    // 3.
    if (e == 0) {
        bool ok = wait_phase(stg_bar, 0, limit, abort_flag, args.status) &&
                  wait_phase_cluster(ready_bar, 0, limit, abort_flag, args.status);
        if (ok)
            for (int p = 0; p < S; ++p)
                if (p != (int)z)
                    ptx::bulk_copy_to_cluster(ptx::mapa(recv + z * block, (uint32_t)p), stg + p * block,
                                              (uint32_t)block, ptx::mapa(recv_bar, (uint32_t)p));
    }
    // 4.
    const bool ok = wait_phase_cluster(recv_bar, 0, limit, abort_flag, args.status) &&
                    wait_phase(stg_bar, 0, limit, abort_flag, args.status);
    if (!__all_sync(0xffffffffu, ok)) return false;
    uint8_t* own = stg_ptr + z * block;
    for (int o = e * 16; o < block; o += 128 * 16) {
        float4 acc = z == 0 ? *reinterpret_cast<const float4*>(own + o)
                            : *reinterpret_cast<const float4*>(recv_ptr + o);
        for (int s = 1; s < S; ++s) {
            const float4 t = s == (int)z ? *reinterpret_cast<const float4*>(own + o)
                                         : *reinterpret_cast<const float4*>(recv_ptr + s * block + o);
            acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
        }
        *reinterpret_cast<float4*>(own + o) = acc;
    }
    ptx::fence_proxy_async_shared();  // visible to the TMA stores
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(sum_bar);
    if (!__all_sync(0xffffffffu, wait_phase(sum_bar, 0, limit, abort_flag, args.status))) return false;
    // 5.
    const int quads = 4 / S, q0 = (int)z * quads;
    if (args.c_tma) {
        if (e < quads * NB) {
            const int qd = q0 + e / NB, bx = e % NB;
            const int64_t y = (int64_t)tm * kBM + qd * 32, x = (int64_t)tn * BN + bx * 32;
            if (y < args.M && x < args.N) {
                ptx::tma_store_2d(tm_c, stg + (qd * NB + bx) * 4096, (int32_t)x, (int32_t)y);
                ptx::bulk_commit();
                ptx::bulk_wait_all();
            }
        }
    } else {
        const bool vec = ((args.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(args.C) & 15) == 0);
        for (int idx = e; idx < quads * 32 * (BN / 4); idx += 128) {
            const int rb = idx / (BN / 4), c4 = idx % (BN / 4);
            const int qd = q0 + rb / 32, rr = rb % 32, bx = c4 / 8, q = c4 % 8;
            const float4 v = *reinterpret_cast<const float4*>(stg_ptr + (qd * NB + bx) * 4096 + rr * 128 +
                                                              ((q ^ (rr & 7)) << 4));
            const int64_t grow = (int64_t)tm * kBM + qd * 32 + rr, gcol = (int64_t)tn * BN + 4 * c4;
            if (grow >= args.M) continue;
            float* dst = args.C + grow * args.ldc + gcol;
            if (vec && gcol + 3 < args.N) {
                *reinterpret_cast<float4*>(dst) = v;
            } else {
                const float w[4] = {v.x, v.y, v.z, v.w};
                for (int k = 0; k < 4 && gcol + k < args.N; ++k) dst[k] = w[k];
            }
        }
    }
    return true;
}

// The epilogue barriers of one warp: the cluster sum's (ready, recv, stg,
// sumd) and this warp's last-arriver load barrier.
struct EpilogueBars {
    uint32_t ready, recv, stg, sumd, fix;
};

// Drain one accumulator buffer of TMEM (this warp's quadrant of the tile) by
// the unit's way out: the cluster K-slice sum, the last-arriver sum of a split
// unit, TMA stores through the idle ring for a CTA's last unit (RING bytes of
// it; a box per 32 columns per warp where they fit), or direct stores.
// false = a bounded wait gave up.
template <int BN, int RING>
__device__ __forceinline__ bool drain_unit(const TcArgs& args, const CUtensorMap* tm_c, const CUtensorMap* tm_p,
                                           const Unit& u, int tm, int tn, uint32_t taddr, int quad, int lane,
                                           bool last_unit, bool clustered, bool fixup, uint32_t ring,
                                           uint8_t* ring_ptr, const EpilogueBars& eb, int64_t limit,
                                           volatile int* abort_flag)
{
    if (clustered)
        return cluster_reduce_store<BN>(args, tm_c, tm, tn, taddr, quad, lane, ring, ring_ptr, eb.ready, eb.recv,
                                        eb.stg, eb.sumd, limit, abort_flag);
    if (fixup && u.slot >= 0 && last_unit)
        return fixup_store<BN>(args, tm_p, tm_c, u, tm, tn, taddr, quad, lane, ring + quad * kFixWarpBytes,
                               ring_ptr + quad * kFixWarpBytes, eb.fix, limit, abort_flag);
    if (last_unit && (u.slot >= 0 || args.c_tma)) {
        constexpr int NBUF = RING / (4 * 4096) < BN / 32 ? RING / (4 * 4096) : BN / 32;
        const uint32_t stg = (uint32_t)(quad * NBUF * 4096);
        if (u.slot < 0)
            store_accumulator_tma<BN, NBUF>(tm_c, (int64_t)tn * BN, (int64_t)tm * kBM + quad * 32, args.N, args.M,
                                            taddr, lane, ring + stg, ring_ptr + stg);
        else
            store_accumulator_tma<BN, NBUF>(tm_p, 0, (int64_t)u.slot * kBM + quad * 32, BN, INT64_MAX, taddr, lane,
                                            ring + stg, ring_ptr + stg);
        return true;
    }
    store_accumulator<BN>(args, u, tm, tn, taddr, quad * 32 + lane);
    return true;
}

// The K-slices of one float4 of a split tile, summed in slice order (so every
// way of summing them gives the same bits), with the loads of up to four
// slices in flight at once (the first, then three at a time).  p: slice 0;
// STRIDE: float4 from one slice to the next.
// COHERENT: loads through L2 only (ld.global.cg), for slices written by other
// CTAs of the same kernel; else the read-only path.
template <int STRIDE, bool COHERENT = false>
__device__ __forceinline__ float4 sum_slices(const float4* __restrict__ p, int splits)
{
    auto ld = [](const float4* q) { return COHERENT ? __ldcg(q) : __ldg(q); };
    float4 acc = ld(p);
    for (int z = 1; z < splits; z += 3) {
        float4 t[3];
#pragma unroll
        for (int i = 0; i < 3; ++i)
            if (z + i < splits) t[i] = ld(p + (int64_t)(z + i) * STRIDE);
#pragma unroll
        for (int i = 0; i < 3; ++i)
            if (z + i < splits) {
                acc.x += t[i].x; acc.y += t[i].y; acc.z += t[i].z; acc.w += t[i].w;
            }
    }
    return acc;
}

// Reduction kernels: 192 threads of at most 42 registers (8 blocks per SM),
// so one block (at most 8064 registers) fits beside a running 448-thread GEMM
// CTA of 128 registers a thread.  Under programmatic serialisation the
// reduction is then resident before the GEMM ends, and the next GEMM's CTAs
// start their setup beside the reduction's last blocks.
constexpr int kReduceThreads = 192;
constexpr int kReduceBlocksPerSm = 8;

// Blocks of a grid-stride reduction over `work` float4: a thread per float4
// (its slices' loads all in flight at once), up to eight full residencies of
// every SM; beyond that the threads loop.
inline int reduce_blocks(int64_t work, int sms)
{
    const int64_t blocks = (work + kReduceThreads - 1) / kReduceThreads;
    const int64_t cap = (int64_t)sms * kReduceBlocksPerSm * 8;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream finishes, and waits for it (griddepcontrol)
// before touching that kernel's output.  cluster > 1: thread-block clusters of
// that many consecutive CTAs (the grid is a multiple of it).
// cooperative: the runtime guarantees that every CTA of the grid is resident
// at once (the launch fails otherwise), for kernels whose CTAs wait on one
// another.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster,
                          bool cooperative, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        if (grid.x % (unsigned)cluster != 0) return cudaErrorInvalidValue;
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = (unsigned)cluster;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    if (cooperative) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeCooperative;
        attr[cfg.numAttrs].val.cooperative = 1;
        ++cfg.numAttrs;
    }
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster,
                       Args&&... args)
{
    return launch_pdl_ex(kern, grid, block, smem, s, cluster, false, std::forward<Args>(args)...);
}

// A barrier across every CTA of a cooperative grid.  bar[0] counts arrivals,
// bar[1] is the generation: a CTA reads the generation, releases its writes
// (fence at GPU scope) and arrives; the last to arrive resets the count and
// advances the generation; the others wait (bounded) until it moves, then
// acquire.  The count is back at zero after every complete barrier; a barrier
// that timed out leaves it as it stands, and the host clears it with the
// status word.  Called by every thread of the CTA (ok_s: a word of the CTA's
// shared memory free for the purpose); false = gave up.
__device__ __forceinline__ bool grid_barrier(unsigned* bar, int64_t limit, int* status, volatile int* ok_s)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        volatile unsigned* gen = bar + 1;
        const unsigned g = *gen;
        __threadfence();
        const unsigned arrived = atomicAdd(bar, 1u) + 1u;
        if (arrived == gridDim.x * gridDim.y * gridDim.z) {
            atomicExch(bar, 0u);
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            const long long t0 = clock64();
            while (*gen == g) {
                if (clock64() - t0 > limit) {
                    atomicExch(status, kStatusTimeout);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        *ok_s = ok;
    }
    __syncthreads();
    return *ok_s != 0;
}

}  // namespace tc

// The in-kernel split kernel for tile width bn and stage depth bk (32 or 16;
// tc_fused.cu); b_presplit: B comes split by the pre-pass (tbhi/tblo) and
// only A is split in the kernel.
cudaError_t tc_fused_main(int bn, int bk, bool b_presplit, const TcPlanState& st, const tc::TcArgs& a,
                          const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbhi,
                          const CUtensorMap& tblo, cudaStream_t s);

// The CTA-pair kernel (tc_pair.cu): 256 x bn tiles, stage depth bk; split
// (kSplitInKernel, kSplitHybrid or kSplitRawA) says which operand pieces come
// from the pre-pass (tbhi, tblo: B; talo: lo of A) and which the kernel's
// converters make; the work in a's dp_tiles / split_tiles counts pair tiles.
// And the sum of its split pair tiles' K-slices.
cudaError_t tc_pair_main(int bn, int bk, int split, const TcPlanState& st, const tc::TcArgs& a,
                         const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbhi,
                         const CUtensorMap& tblo, const CUtensorMap& talo, cudaStream_t s);
cudaError_t tc_pair_reduce(int bn, const TcPlanState& st, const tc::TcArgs& a, cudaStream_t s);
// The CTA-pair kernel with A in tensor memory (256 x 256 tiles, 32-k stages):
// A read from the caller's A by TMA (ta: 16-byte aligned rows) and split by
// the kernel's loader warps, hi and lo of B by the pre-pass (tbhi, tblo).
cudaError_t tc_pair_tmem_main(const TcPlanState& st, const tc::TcArgs& a, const CUtensorMap& ta,
                              const CUtensorMap& tbhi, const CUtensorMap& tblo, cudaStream_t s);

}  // namespace gemm_f32
