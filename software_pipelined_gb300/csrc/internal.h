// Internal interfaces between the C-ABI layer (api.cu) and the kernel files.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/gemm_f32.h"

namespace gemm_f32 {

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device (the attribute belongs to the device's context).
// `done` is one bit per device ordinal (< 64), kept by the caller per kernel.
template <typename Kernel>
inline cudaError_t smem_limit_once(Kernel kern, int bytes, std::atomic<uint64_t>& done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// ---- SIMT FFMA kernel (simt_gemm.cu) --------------------------------------
struct SimtConfig {
    int bm, bn, bk;   // CTA tile
    int tm, tn;       // per-thread register tile
    int stages;       // cp.async ring depth (1 = single buffer, 2 = double, ...)
    bool sep;         // A and B published by separate barriers (ablation)
    int ksl = 1;      // K-slice groups inside the CTA (sliced K)
    bool shfl = false; // fragments handed out by warp shuffles (ablation), not broadcast loads
};
// Configurations compiled into the library; `id` indexes this table.
int simt_num_configs();
const SimtConfig& simt_config(int id);
// bk = 0: the first compiled K-tile depth for that tile and ring.  -1 if none.
int simt_find_config(int bm, int bn, int stages, bool sep = false, int bk = 0, int ksl = 1, bool shfl = false);

struct SimtArgs {
    int64_t M, N, K;
    const float* A; int64_t lda;
    const float* B; int64_t ldb;
    float* C; int64_t ldc;
    int split_k;          // >1: write partials to `partial`
    int64_t k_chunk;      // K per split (multiple of bk)
    float* partial;       // split_k x M x ldp
    int64_t ldp;
    // Strided batch (split_k == 1): grid z runs `batch` independent products,
    // problem z at A + z*stride_a, B + z*stride_b, C + z*stride_c.
    int64_t batch = 1;
    int64_t stride_a = 0, stride_b = 0, stride_c = 0;
};
cudaError_t simt_launch(int config_id, const SimtArgs& a, cudaStream_t s);

// ---- short-M kernel (rows.cu) ----------------------------------------------
// C = A*B for M <= kRowsMaxM, streaming B once; K in ranges of `range` rows
// (rows_range: a multiple of 256), each range's partial written to `partial`
// (range z at partial + z*M*ldp) for the split-K reduction when K spans more
// than one range, else C directly.
constexpr int64_t kRowsMaxM = 16;
struct RowsArgs {
    int64_t M, N, K;
    const float* A; int64_t lda;
    const float* B; int64_t ldb;
    float* C; int64_t ldc;
    float* partial; int64_t ldp;
    int64_t range;
};
int64_t rows_range(int64_t N, int64_t K, int sms);
cudaError_t rows_launch(const RowsArgs& a, cudaStream_t s);
// C = A*B for N <= kColsMaxN, streaming A once (a warp per row of C; rows.cu).
constexpr int64_t kColsMaxN = 16;
struct ColsArgs {
    int64_t M, N, K;
    const float* A; int64_t lda;
    const float* B; int64_t ldb;
    float* C; int64_t ldc;
};
cudaError_t cols_launch(const ColsArgs& a, int sms, cudaStream_t s);

// Deterministic split-K reduction: C[i][j] = sum_{z=0}^{splits-1} P[z][i][j]
// in ascending z (splitk_reduce.cu).
cudaError_t splitk_reduce_launch(const float* P, int splits, int64_t M, int64_t N, int64_t ldp,
                                 float* C, int64_t ldc, cudaStream_t s);
// C = 0 (the K == 0 case).
cudaError_t zero_fill_launch(float* C, int64_t M, int64_t N, int64_t ldc, cudaStream_t s);

// ---- tcgen05 3xTF32 kernel (tc_gemm.cu) -----------------------------------
struct TcConfig {
    int bm, bn, bk;  // tile (bm = 128 rows = TMEM lanes, or 256 for a CTA pair; bk = 32 fp32 = 128 B)
    int stages;      // smem ring depth
    bool sep;        // separate full barriers for A and B (ablation)
    int split;       // where the 3xTF32 split happens: kSplitPrepass, kSplitInKernel, kSplitHybrid, kSplitRawA
};
enum : int {
    kSplitPrepass = 0,   // a pre-pass writes hi/lo of A and B to scratch
    kSplitInKernel = 1,  // raw A and B by TMA, split by converter warps
    kSplitHybrid = 2,    // raw A split in the kernel, B split by the pre-pass
    kSplitRawA = 3,      // hi of A read from A (truncated by the MMA); the pre-pass writes lo of A, hi/lo of B
    kSplitTmemA = 4      // CTA pairs only: A split by the kernel's loader warps into tensor memory, B by the pre-pass
};
int tc_num_configs();
const TcConfig& tc_config(int id);
int tc_find_config(int bn, int stages, bool sep, int split, int bk = 0);
// The CTA-pair configuration (256-row tiles) of tile width bn, stage depth bk
// (0 = 32) and split mode (kSplitInKernel; kSplitHybrid: B by the pre-pass;
// kSplitRawA: lo of A and B by the pre-pass; kSplitTmemA: A into tensor
// memory by the kernel, B by the pre-pass), or -1.
int tc_find_pair_config(int bn, int bk, int split = kSplitInKernel);
// How many pairs of that configuration run at once on this device (0 when the
// occupancy query fails).
int tc_pair_slots(int bn, int bk, int sms, int split = kSplitInKernel);

// Plan-time state of the tensor-core path: split-operand scratch and the
// tensor maps that describe it, and the work decomposition.
//
// The output tiles are taken in the kernel's tile order.  The first dp_tiles
// are computed whole and written straight to C.  The remaining split_tiles are
// computed as `splits` K-slices each, written as dense 128 x BN partial tiles to
// `partial`, and summed in slice order by the tile reduction.  With a global
// split-K request every tile is a split tile; with the automatic policy only
// the tiles of a partial last wave are split, so that they finish in a
// fraction of a tile's time instead of leaving most SMs idle.
struct TcPlanState {
    int config_id = -1;
    int terms = 3;
    int64_t kp = 0;            // padded K (row length of split operands), multiple of 32
    int tiles_m = 0, tiles_n = 0;
    int dp_tiles = 0;
    int split_tiles = 0;
    int splits = 1;            // K-slices per split tile
    int kb_per_split = 0;      // k-blocks of 32 per slice
    float* a_hi = nullptr;     // M x kp
    float* a_lo = nullptr;
    float* b_hi = nullptr;     // N x kp (B transposed: K-major)
    float* b_lo = nullptr;
    float* partial = nullptr;  // split_tiles x splits x 128 x BN
    size_t partial_bytes = 0;
    alignas(64) unsigned char tmap_a_hi[128];
    alignas(64) unsigned char tmap_a_lo[128];
    alignas(64) unsigned char tmap_b_hi[128];
    alignas(64) unsigned char tmap_b_lo[128];
    int num_sms = 0;
    int64_t timeout_cycles = 0;
    int withhold_stage = 0;
    int tile_group = 0;        // tile-rows per raster group (0 = default)
    int split_request = 0;     // the split policy tc_configure was given
    // K-slice sums (the plan's split_reduce option): 0 and 1 = the reduction
    // kernel; 2 = in a thread-block cluster where possible; 3 = the last slice
    // to arrive sums the tile where possible; 4 = the CTA pairs' whole grid,
    // after a grid-wide barrier
    int cluster_mode = 0;
    int cluster = 0;           // > 1: slices per tile, summed in a thread-block cluster
    int fixup = 0;             // 1: the last slice to arrive sums the tile
    int gridsum = 0;           // 1: CTA pairs: the whole (cooperative) grid sums the slices
                               // after a grid-wide barrier, no reduction launch
    int* sem = nullptr;        // fixup arrival counters or the grid barrier's count and
                               // generation (zero between runs), sem_bytes long
    size_t sem_bytes = 0;
    // In-kernel and hybrid split plans: the pre-split configuration of the same
    // tile width, used when a base pointer of A or B is not 16-byte aligned;
    // tensor maps over the caller's raw A and B, re-encoded when they change.
    int fallback_config_id = -1;
    int pair_slots = 0;        // CTA-pair plans: pairs of CTAs resident at once
    mutable const float* raw_a = nullptr;
    mutable const float* raw_b = nullptr;
    alignas(64) mutable unsigned char tmap_a_raw[128];
    alignas(64) mutable unsigned char tmap_b_raw[128];
    // TMA-store maps: the partial-tile buffer (set with tc_set_partial) and the
    // caller's C (re-encoded when C moves; c_tma = 0 when C cannot take TMA
    // stores: base not 16-byte aligned, or ldc or N not a multiple of 4)
    alignas(64) unsigned char tmap_p[128];
    alignas(64) mutable unsigned char tmap_c[128];
    mutable float* c_ptr = nullptr;
    mutable int c_tma = 0;
};
// Work decomposition for config t.config_id: split_request 0 = automatic
// (split the tiles of a partial last wave), 1 = none, >= 2 = every tile in that
// many K-slices.  Sets kp, tiles, dp/split tiles, splits and partial_bytes.
void tc_configure(TcPlanState& t, int64_t M, int64_t N, int64_t K, int split_request);
// Allocates nothing: encodes tensor maps over already-allocated split buffers
// (and over st.partial when set).
cudaError_t tc_prepare(TcPlanState& st, int64_t M, int64_t N, int64_t K);
// Point the state's split units at `partial` (partial_bytes long) and encode
// the TMA-store map over it.
cudaError_t tc_set_partial(TcPlanState& st, float* partial);
// Row panels of a plan, for the pipelined host-buffer path: `out` becomes the
// plan's state re-configured for rows [r0, r0 + mp) of A and C (A, B: the
// device buffers the panels read); its partial-tile buffer is left NULL for
// the caller to provide (out.partial_bytes long).
cudaError_t tc_panel_prepare(const TcPlanState& full, int64_t r0, int64_t mp, int64_t N, int64_t K,
                             const float* A, int64_t lda, const float* B, int64_t ldb, TcPlanState& out);
// A block of rows r0..r0+mp and columns c0..c0+nq of the product (c0 and nq
// whole tiles): the panel state over those rows, with the block's rows of the
// split B and the block's columns of the raw B.  The block's split B is
// written by tc_split_b on this state with B + c0 and N = nq.
cudaError_t tc_block_prepare(const TcPlanState& full, int64_t r0, int64_t mp, int64_t c0, int64_t nq, int64_t K,
                             const float* A, int64_t lda, const float* B, int64_t ldb, TcPlanState& out);
// The B part of the pre-pass for the whole plan (when its route needs it).
cudaError_t tc_split_b(const TcPlanState& full, int64_t N, int64_t K, const float* A, const float* B,
                       int64_t ldb, cudaStream_t s);
// One panel: its A rows' pre-pass (when the route needs one and pre_a is set;
// the column blocks of one panel share their rows' split A, so only the first
// block runs it), the GEMM, the reduction.
cudaError_t tc_panel_run(const TcPlanState& panel, int64_t mp, int64_t N, int64_t K, const float* A_panel,
                         int64_t lda, const float* B, int64_t ldb, float* C_panel, int64_t ldc, int* status,
                         cudaStream_t s, bool pre_a = true);
// ev: NULL, or four events recorded before the split, before the main kernel,
// after the main kernel and after the split-K reduction.
cudaError_t tc_launch(const TcPlanState& st, int64_t M, int64_t N, int64_t K,
                      const float* A, int64_t lda, const float* B, int64_t ldb,
                      float* C, int64_t ldc, int* status, cudaStream_t s,
                      cudaEvent_t* ev = nullptr);

// Device status word values written by kernels.
enum : int { kStatusOk = 0, kStatusTimeout = 1 };

}  // namespace gemm_f32
