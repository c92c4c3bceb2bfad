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

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream finishes, and waits for it (griddepcontrol)
// before touching that kernel's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace tc

// The in-kernel split kernel for tile width bn (tc_fused.cu); b_presplit: B
// comes split by the pre-pass (tbhi/tblo) and only A is split in the kernel.
cudaError_t tc_fused_main(int bn, bool b_presplit, const TcPlanState& st, const tc::TcArgs& a,
                          const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbhi,
                          const CUtensorMap& tblo, cudaStream_t s);

}  // namespace gemm_f32
