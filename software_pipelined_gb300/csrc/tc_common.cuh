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
    int cluster;         // > 1: every tile split in `cluster` K-slices, one CTA each, the
                         // slices of a tile one thread-block cluster that sums them
                         // through distributed shared memory (no partial tiles)
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

// Epilogue through TMA stores, for a CTA's last unit (its operand ring is then
// idle and serves as staging).  The calling warp owns TMEM lanes = tile rows
// y0 .. y0+31 of the destination (C, or the partial-tile buffer) and the 8 KB
// of staging at `stage` (two 4 KB boxes of 32 rows x 32 FP32 in the 128-byte
// swizzled layout: 16-byte chunk q of row r at chunk q ^ (r % 8), so the 8
// lanes of each store phase hit 8 different chunks).  Per 32 columns: two
// TMEM loads, 8 conflict-free 16-byte shared stores per lane, one TMA store
// of the box (clipped at the tensor's edge; boxes wholly past it are skipped).
template <int BN>
__device__ __forceinline__ void store_accumulator_tma(const CUtensorMap* map, int64_t x0, int64_t y0,
                                                      int64_t xlim, int64_t ylim, uint32_t taddr, int lane,
                                                      uint32_t stage, uint8_t* stage_ptr)
{
    // Only boxes that are stored are staged, so every staged box is one
    // committed group and "at most one group still reading" below means the
    // store of the box two back (the same buffer) is done with it.
    const int cols = y0 < ylim ? (int)(xlim - x0 < BN ? xlim - x0 : BN) : 0;
#pragma unroll 1
    for (int c = 0; c < cols; c += 32) {
        const int b = (c >> 5) & 1;
        if (c >= 64) {
            // box b was stored two boxes ago: its store must be done reading
            if (lane == 0) ptx::bulk_wait_read<1>();
            __syncwarp();
        }
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x16(taddr + c, *reinterpret_cast<uint32_t(*)[16]>(r));
        ptx::tmem_ld_32x32b_x16(taddr + c + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
        ptx::tmem_wait_ld();
        uint8_t* row = stage_ptr + b * 4096 + lane * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(row + ((q ^ (lane & 7)) << 4)) =
                make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        ptx::fence_proxy_async_shared();  // generic-proxy writes -> the TMA engine's reads
        __syncwarp();
        if (lane == 0) {
            ptx::tma_store_2d(map, stage + b * 4096, (int32_t)(x0 + c), (int32_t)y0);
            ptx::bulk_commit();
        }
    }
    if (lane == 0) ptx::bulk_wait_all();  // complete before the staging is reused or freed
    __syncwarp();
}

// Epilogue of a K-sliced tile whose S = args.cluster slices are the S CTAs of
// one cluster (rank z = slice z).  Rows are owned in blocks: rank r sums rows
// r*128/S .. (r+1)*128/S - 1 of the tile.  Called by the 128 epilogue threads
// (thread = TMEM lane = tile row) once this CTA's accumulator is complete.
//   1. This CTA's MMAs are done, so its operand ring is idle: one thread
//      arrives on every rank's `ready` barrier.
//   2. Wait until all S rings are idle (`ready` complete: S arrivals).
//   3. Each thread sends its row (BN FP32, from TMEM) into slice z's row of
//      the owner's receive buffer, laid over the owner's idle ring
//      ([S][128/S][BN + 4] FP32; the 4-float pad spreads the rows of a warp
//      over the banks), then arrives on the owner's `recv` barrier.
//   4. Wait for the 128 rows this CTA owns (`recv` complete: 128 arrivals),
//      sum the S slices in slice order (the order of the reduction kernel, so
//      the result is the same bit for bit) and store them to C.
// Every wait is bounded; false means a wait gave up (status already set).  No
// CTA leaves the kernel before the cluster barrier at its end, so no remote
// access ever targets a CTA that has exited.
template <int BN>
__device__ bool cluster_reduce_store(const TcArgs& args, int tm, int tn, uint32_t taddr, int row,
                                     uint32_t recv_addr, const float* recv_ptr, uint32_t ready_bar,
                                     uint32_t recv_bar, int64_t limit, volatile int* abort_flag)
{
    constexpr int LD = BN + 4;
    const int S = args.cluster;
    const int rows_per = kBM / S;
    const uint32_t z = ptx::cluster_ctarank();
    if (row == 0)
        for (int r = 0; r < S; ++r) ptx::mbar_arrive_cluster(ptx::mapa(ready_bar, (uint32_t)r));
    // warp-uniform outcome: the TMEM loads below are warp-collective
    if (!__all_sync(0xffffffffu, wait_phase_cluster(ready_bar, 0, limit, abort_flag, args.status))) return false;
    const uint32_t owner = (uint32_t)(row / rows_per);
    const uint32_t dst = ptx::mapa(recv_addr, owner) +
                         (uint32_t)(((int)z * rows_per + row % rows_per) * LD) * 4u;
#pragma unroll 1
    for (int c = 0; c < BN; c += 16) {
        uint32_t r[16];
        ptx::tmem_ld_32x32b_x16(taddr + c, r);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; j += 4)
            ptx::st_cluster_v4(dst + (uint32_t)(c + j) * 4u, r[j], r[j + 1], r[j + 2], r[j + 3]);
    }
    ptx::mbar_arrive_cluster(ptx::mapa(recv_bar, owner));
    if (!__all_sync(0xffffffffu, wait_phase_cluster(recv_bar, 0, limit, abort_flag, args.status))) return false;
    const bool vec = ((args.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(args.C) & 15) == 0);
    const int row0 = tm * kBM + (int)z * rows_per;
    for (int idx = row; idx < rows_per * (BN / 4); idx += kBM) {
        const int r = idx / (BN / 4), c4 = idx % (BN / 4);
        float4 acc = *reinterpret_cast<const float4*>(recv_ptr + r * LD + 4 * c4);
        for (int s = 1; s < S; ++s) {
            const float4 t = *reinterpret_cast<const float4*>(recv_ptr + (s * rows_per + r) * LD + 4 * c4);
            acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
        }
        const int64_t grow = (int64_t)row0 + r, gcol = (int64_t)tn * BN + 4 * c4;
        if (grow >= args.M) continue;
        float* dst_c = args.C + grow * args.ldc + gcol;
        if (vec && gcol + 3 < args.N) {
            *reinterpret_cast<float4*>(dst_c) = acc;
        } else {
            const float v[4] = {acc.x, acc.y, acc.z, acc.w};
            for (int q = 0; q < 4 && gcol + q < args.N; ++q) dst_c[q] = v[q];
        }
    }
    return true;
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream finishes, and waits for it (griddepcontrol)
// before touching that kernel's output.  cluster > 1: thread-block clusters of
// that many consecutive CTAs (the grid is a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        if (grid.x % (unsigned)cluster != 0) return cudaErrorInvalidValue;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace tc

// The in-kernel split kernel for tile width bn (tc_fused.cu); b_presplit: B
// comes split by the pre-pass (tbhi/tblo) and only A is split in the kernel.
cudaError_t tc_fused_main(int bn, bool b_presplit, const TcPlanState& st, const tc::TcArgs& a,
                          const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbhi,
                          const CUtensorMap& tblo, cudaStream_t s);

}  // namespace gemm_f32
