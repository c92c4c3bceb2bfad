// Host side of the tcgen05 3xTF32 GEMM: the configuration table, the work
// decomposition of a plan (whole tiles and K-sliced tiles of the last wave),
// the tensor maps, and the launch sequence of one run (operand pre-pass, main
// kernel, split-tile reduction), whole or by row panels.  The kernels are in
// tc_kernels.cuh.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tc_kernels.cuh"

namespace gemm_f32 {
namespace {

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

// 2-D tensor map over a rows x kp K-major FP32 buffer, box {box_k, box_rows}:
// rows of 32 FP32 in the 128-byte swizzle, of 16 in the 64-byte one; zero fill
// outside.
cudaError_t encode_kmajor(void* out, float* base, int64_t rows, int64_t kp, int box_rows, int box_k = kBK)
{
    EncodeFn enc = get_encode();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)kp, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(kp * 4)};
    cuuint32_t box[2] = {(cuuint32_t)box_k, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     box_k == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Row-major FP32 matrix (rows x cols, leading dimension ld) as the target of
// TMA stores of 32 x 32 boxes in the 128-byte swizzled layout.
cudaError_t encode_store_map(void* out, float* base, int64_t rows, int64_t cols, int64_t ld)
{
    EncodeFn enc = get_encode();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 4)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int grid_cap(int64_t work, int sms)
{
    const int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

// Tensor maps over the caller's raw operands for the in-kernel split: A (M x K,
// lda) as K-major boxes {32, 128}; B (K x N, ldb) as boxes of 32 columns x 32
// rows.  Both 128-byte swizzled with zero fill; need 16-byte aligned rows.
cudaError_t encode_raw_a(void* out, const float* A, int64_t M, int64_t K, int64_t lda, int box_k)
{
    EncodeFn enc = get_encode();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(lda * 4)};
    cuuint32_t box[2] = {(cuuint32_t)box_k, (cuuint32_t)kBM};
    cuuint32_t estr[2] = {1, 1};
    // rows of 32 FP32 in the 128-byte swizzle, of 16 in the 64-byte one
    CUresult r = enc(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                     const_cast<float*>(A), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     box_k == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_raw_b(void* out, const float* B, int64_t K, int64_t N, int64_t ldb, int box_k)
{
    EncodeFn enc = get_encode();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)K};
    cuuint64_t strides[1] = {(cuuint64_t)(ldb * 4)};
    cuuint32_t box[2] = {32, (cuuint32_t)box_k};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                     const_cast<float*>(B), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int BN, int STAGES, bool SEP = false>
cudaError_t launch_main(const TcPlanState& st, const TcArgs& a, const void* tmap_a_hi, cudaStream_t s)
{
    using L = TcLayout<BN, STAGES>;
    auto kern = tc_gemm_kernel<BN, STAGES, SEP>;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = smem_limit_once(kern, L::SMEM_BYTES, smem_set); e != cudaSuccess) return e;
    const int work = a.dp_tiles + a.split_tiles * a.splits;
    const int grid = work < st.num_sms ? work : st.num_sms;
    static_assert(L::RING_BYTES >= 4 * 8192, "the ring holds the TMA-store staging");
    if ((a.cluster > 1 && !L::CLUSTER_OK) || (a.fixup && !L::FIXUP_OK)) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), L::SMEM_BYTES, s, a.cluster,
                      *reinterpret_cast<const CUtensorMap*>(tmap_a_hi),
                      *reinterpret_cast<const CUtensorMap*>(st.tmap_a_lo),
                      *reinterpret_cast<const CUtensorMap*>(st.tmap_b_hi),
                      *reinterpret_cast<const CUtensorMap*>(st.tmap_b_lo),
                      *reinterpret_cast<const CUtensorMap*>(st.tmap_c),
                      *reinterpret_cast<const CUtensorMap*>(st.tmap_p), a);
}

template <int BN>
cudaError_t launch_reduce(const TcPlanState& st, const TcArgs& a, cudaStream_t s)
{
    const int64_t total = (int64_t)a.split_tiles * kBM * (BN / 4);
    return launch_pdl(tile_reduce_kernel<BN>, dim3(reduce_blocks(total, st.num_sms)), dim3(kReduceThreads), 0, s, 1,
                      reinterpret_cast<const float4*>(a.partial), a.dp_tiles, a.split_tiles, a.splits,
                      a.tiles_m, a.tiles_n, a.group, a.M, a.N, a.C, a.ldc);
}

template <int BN>
cudaError_t launch_pair_reduce(const TcPlanState& st, const TcArgs& a, cudaStream_t s)
{
    return tc_pair_reduce(BN, st, a, s);
}

using MainFn = cudaError_t (*)(const TcPlanState&, const TcArgs&, const void*, cudaStream_t);
using LaunchFn = cudaError_t (*)(const TcPlanState&, const TcArgs&, cudaStream_t);
struct TcEntry {
    TcConfig cfg;
    MainFn main;      // NULL where the split happens in the kernel (tc_fused_main)
    LaunchFn reduce;
    bool cluster_ok;  // the ring can hold the cluster reduction's receive buffer
    bool fixup_ok;    // the ring can hold the last-arriver sum's staging
};
template <int BN, int STAGES>
constexpr bool kClusterOk = TcLayout<BN, STAGES>::CLUSTER_OK;
template <int BN, int STAGES>
constexpr bool kFixupOk = TcLayout<BN, STAGES>::FIXUP_OK;
const TcEntry kTc[] = {
    // the ring as deep as shared memory allows, per tile width
    {{128, 128, 32, 3, false, kSplitPrepass}, launch_main<128, 3>, launch_reduce<128>, kClusterOk<128, 3>, kFixupOk<128, 3>},
    {{128, 256, 32, 2, false, kSplitPrepass}, launch_main<256, 2>, launch_reduce<256>, kClusterOk<256, 2>, kFixupOk<256, 2>},
    {{128, 64, 32, 4, false, kSplitPrepass}, launch_main<64, 4>, launch_reduce<64>, kClusterOk<64, 4>, kFixupOk<64, 4>},
    // pipeline-depth ablation: single-buffered (1) and shallower rings
    {{128, 256, 32, 1, false, kSplitPrepass}, launch_main<256, 1>, launch_reduce<256>, kClusterOk<256, 1>, kFixupOk<256, 1>},
    {{128, 128, 32, 1, false, kSplitPrepass}, launch_main<128, 1>, launch_reduce<128>, kClusterOk<128, 1>, kFixupOk<128, 1>},
    {{128, 128, 32, 2, false, kSplitPrepass}, launch_main<128, 2>, launch_reduce<128>, kClusterOk<128, 2>, kFixupOk<128, 2>},
    {{128, 64, 32, 2, false, kSplitPrepass}, launch_main<64, 2>, launch_reduce<64>, kClusterOk<64, 2>, kFixupOk<64, 2>},
    // barrier-coalescing ablation: separate full barriers for A and B
    {{128, 256, 32, 2, true, kSplitPrepass}, launch_main<256, 2, true>, launch_reduce<256>, kClusterOk<256, 2>, kFixupOk<256, 2>},
    {{128, 128, 32, 3, true, kSplitPrepass}, launch_main<128, 3, true>, launch_reduce<128>, kClusterOk<128, 3>, kFixupOk<128, 3>},
    // operands split inside the kernel (stages = MMA-facing slots; the fused
    // kernel's 3 x 64 KB ring holds the cluster sum's 128 KB, its 2 x 96 KB
    // ring of 128 x 256 tiles not the 256 KB those would need)
    {{128, 128, 32, 3, false, kSplitInKernel}, nullptr, launch_reduce<128>, true, true},
    {{128, 256, 32, 2, false, kSplitInKernel}, nullptr, launch_reduce<256>, false, true},
    // the same with half-size (16-k) stages, twice as deep: 6 x 32 KB, 4 x 48 KB
    {{128, 128, 16, 6, false, kSplitInKernel}, nullptr, launch_reduce<128>, true, true},
    {{128, 256, 16, 4, false, kSplitInKernel}, nullptr, launch_reduce<256>, false, true},
    // A split inside the kernel, B by the pre-pass
    {{128, 128, 32, 3, false, kSplitHybrid}, nullptr, launch_reduce<128>, true, true},
    {{128, 256, 32, 2, false, kSplitHybrid}, nullptr, launch_reduce<256>, false, true},
    // hi of A read from the caller's A, lo of A and both pieces of B by the pre-pass
    {{128, 128, 32, 3, false, kSplitRawA}, launch_main<128, 3>, launch_reduce<128>, kClusterOk<128, 3>, kFixupOk<128, 3>},
    {{128, 256, 32, 2, false, kSplitRawA}, launch_main<256, 2>, launch_reduce<256>, kClusterOk<256, 2>, kFixupOk<256, 2>},
    // CTA pairs (tc_pair.cu): 256 x BN tiles, operands split in the kernel,
    // each CTA holding its 128 rows of A and half of B; rings of 192 KB
    {{256, 256, 32, 3, false, kSplitInKernel}, nullptr, launch_pair_reduce<256>, false, false},
    {{256, 256, 16, 6, false, kSplitInKernel}, nullptr, launch_pair_reduce<256>, false, false},
    {{256, 128, 32, 4, false, kSplitInKernel}, nullptr, launch_pair_reduce<128>, false, false},
    {{256, 128, 16, 8, false, kSplitInKernel}, nullptr, launch_pair_reduce<128>, false, false},
    // CTA pairs with B split by the pre-pass (each CTA loads its half of hi_B
    // and lo_B), only lo_A computed in the kernel
    {{256, 256, 32, 3, false, kSplitHybrid}, nullptr, launch_pair_reduce<256>, false, false},
    {{256, 128, 32, 4, false, kSplitHybrid}, nullptr, launch_pair_reduce<128>, false, false},
    // CTA pairs with lo of A and both pieces of B by the pre-pass, hi of A read
    // from A: no conversion between a stage's copy and its MMAs
    {{256, 256, 32, 3, false, kSplitRawA}, nullptr, launch_pair_reduce<256>, false, false},
    {{256, 256, 16, 6, false, kSplitRawA}, nullptr, launch_pair_reduce<256>, false, false},
    {{256, 128, 32, 4, false, kSplitRawA}, nullptr, launch_pair_reduce<128>, false, false},
    // CTA pairs with A split by the kernel's loader warps into tensor memory
    // and hi/lo of B by the pre-pass: 5 B stages, raw A staged 3 deep
    {{256, 256, 32, 5, false, kSplitTmemA}, nullptr, launch_pair_reduce<256>, false, false},
};

}  // namespace

int tc_num_configs() { return (int)(sizeof(kTc) / sizeof(kTc[0])); }
const TcConfig& tc_config(int id) { return kTc[id].cfg; }
int tc_find_config(int bn, int stages, bool sep, int split, int bk)
{
    for (int i = 0; i < tc_num_configs(); ++i) {
        const TcConfig& c = kTc[i].cfg;
        if (c.bm == kBM && c.bn == bn && (stages == 0 || c.stages == stages) && c.sep == sep && c.split == split &&
            (bk == 0 || c.bk == bk))
            return i;
    }
    return -1;
}

int tc_find_pair_config(int bn, int bk, int split)
{
    for (int i = 0; i < tc_num_configs(); ++i) {
        const TcConfig& c = kTc[i].cfg;
        if (c.bm == 2 * kBM && c.bn == bn && c.bk == (bk ? bk : kBK) && c.split == split) return i;
    }
    return -1;
}

namespace {

// The work of a CTA-pair plan, in pair tiles (two tile rows of one tile
// column): the same policy as below with a pair tile for a tile and the pairs
// resident at once for the SMs.  tiles_m counts 128-row tiles, rounded up to
// whole pairs (the second tile of the last pair may lie past M: its rows are
// computed from TMA's zero fill and never stored).
void pair_configure(TcPlanState& t, int64_t M, int64_t N, int split_request)
{
    const TcConfig& c = kTc[t.config_id].cfg;
    const int num_kb = (int)(t.kp / kBK);
    t.tiles_m = 2 * (int)((M + 2 * kBM - 1) / (2 * kBM));
    t.tiles_n = (int)((N + c.bn - 1) / c.bn);
    const int ptiles = t.tiles_m / 2 * t.tiles_n;
    const int wave = t.pair_slots > 0 ? t.pair_slots : (t.num_sms > 1 ? t.num_sms / 2 : 1);
    t.dp_tiles = ptiles;
    t.split_tiles = 0;
    t.splits = 1;
    int want = 1;
    if (split_request >= 2) {
        want = split_request;
        t.dp_tiles = 0;
        t.split_tiles = ptiles;
    } else if (split_request == 0 && ptiles > wave && ptiles % wave != 0) {
        const int rem = ptiles % wave;
        want = std::min(std::min(wave / rem, 8), num_kb / 4);
        if (want >= 2) {
            t.dp_tiles = ptiles - rem;
            t.split_tiles = rem;
        }
    }
    if (t.split_tiles > 0) {
        if (want > num_kb) want = num_kb;
        const int kb_per = (num_kb + want - 1) / want;
        const int splits = (num_kb + kb_per - 1) / kb_per;
        if (splits < 2) {
            t.dp_tiles = ptiles;
            t.split_tiles = 0;
        } else {
            t.splits = splits;
            t.kb_per_split = kb_per;
        }
    }
    if (t.split_tiles == 0) t.kb_per_split = num_kb;
    // Every tile in 2 or 4 K-slices: with the cluster sum asked for, the S
    // pairs of a tile run as one cluster and sum the slices in distributed
    // shared memory (no partial tiles, no reduction launch).
    t.cluster = t.cluster_mode == 2 && t.dp_tiles == 0 && t.split_tiles > 0 && (t.splits == 2 || t.splits == 4)
                    ? t.splits : 0;
    t.fixup = 0;
    // With the grid sum asked for, the pairs' whole (cooperative) grid sums
    // the slices after a grid-wide barrier (no reduction launch); not in the
    // tensor-memory form.
    t.gridsum = t.cluster_mode == 4 && t.split_tiles > 0 && !t.cluster && c.split != kSplitTmemA;
    t.sem_bytes = t.gridsum ? 2 * sizeof(int) : 0;
    t.partial_bytes = t.split_tiles && !t.cluster ? size_t(2) * t.split_tiles * t.splits * kBM * c.bn * sizeof(float)
                                                 : 0;
}

}  // namespace

void tc_configure(TcPlanState& t, int64_t M, int64_t N, int64_t K, int split_request)
{
    const TcConfig& c = kTc[t.config_id].cfg;
    t.split_request = split_request;
    if (c.bm == 2 * kBM) {
        t.kp = (K + kBK - 1) / kBK * kBK;
        pair_configure(t, M, N, split_request);
        return;
    }
    t.kp = (K + kBK - 1) / kBK * kBK;
    const int num_kb = (int)(t.kp / kBK);
    t.tiles_m = (int)((M + kBM - 1) / kBM);
    t.tiles_n = (int)((N + c.bn - 1) / c.bn);
    const int tiles = t.tiles_m * t.tiles_n;
    const int sms = t.num_sms > 0 ? t.num_sms : 1;
    t.dp_tiles = tiles;
    t.split_tiles = 0;
    t.splits = 1;
    int want = 1;
    if (split_request >= 2) {
        // every tile in split_request K-slices
        want = split_request;
        t.dp_tiles = 0;
        t.split_tiles = tiles;
    } else if (split_request == 0 && tiles > sms && tiles % sms != 0) {
        // split the tiles of the partial last wave so they fill the machine once
        const int rem = tiles % sms;
        want = sms / rem;
        if (want > 8) want = 8;
        if (want > num_kb / 4) want = num_kb / 4;
        if (want >= 2) {
            t.dp_tiles = tiles - rem;
            t.split_tiles = rem;
        }
    }
    if (t.split_tiles > 0) {
        if (want > num_kb) want = num_kb;
        int kb_per = (num_kb + want - 1) / want;
        int splits = (num_kb + kb_per - 1) / kb_per;  // no empty slice
        if (splits < 2) {
            t.dp_tiles = tiles;
            t.split_tiles = 0;
        } else {
            t.splits = splits;
            t.kb_per_split = kb_per;
        }
    }
    if (t.split_tiles == 0) t.kb_per_split = num_kb;
    // Every tile in 2 or 4 slices, one CTA per slice, all at once: the slices
    // of a tile can run as one thread-block cluster that sums them in
    // distributed shared memory (no partial tiles, no reduction launch).
    t.cluster = 0;
    const bool cluster_fits = kTc[t.config_id].cluster_ok && t.dp_tiles == 0 && t.split_tiles > 0 &&
                              (t.splits == 2 || t.splits == 4) && t.split_tiles * t.splits <= sms;
    if (cluster_fits && t.cluster_mode == 2) t.cluster = t.splits;
    // Split units that are all their CTA's last unit (at most one wave of
    // them) and at most 8 slices: the last slice to arrive sums the tile.
    t.fixup = 0;
    const bool fixup_fits = kTc[t.config_id].fixup_ok && t.split_tiles > 0 && t.splits <= 8 &&
                            t.split_tiles * t.splits <= sms && !t.cluster;
    if (fixup_fits && t.cluster_mode == 3) t.fixup = 1;
    t.gridsum = 0;  // CTA pairs only
    t.sem_bytes = t.fixup ? size_t(t.split_tiles) * 4 * sizeof(int) : 0;
    t.partial_bytes = t.split_tiles && !t.cluster ? size_t(t.split_tiles) * t.splits * kBM * c.bn * sizeof(float)
                                                  : 0;
}

cudaError_t tc_set_partial(TcPlanState& st, float* partial)
{
    st.partial = partial;
    if (!partial || st.partial_bytes == 0) return cudaSuccess;
    const int64_t bn = kTc[st.config_id].cfg.bn;
    return encode_store_map(st.tmap_p, partial, (int64_t)(st.partial_bytes / (bn * sizeof(float))), bn, bn);
}

// k per box of the pre-split operands' tensor maps: a pair plan loads them in
// its own stage depth, the one-CTA kernels in 32-k blocks.
static int split_box_k(const TcConfig& c) { return c.bm == 2 * kBM ? c.bk : kBK; }

cudaError_t tc_prepare(TcPlanState& st, int64_t M, int64_t N, int64_t K)
{
    (void)K;
    const TcConfig& c = kTc[st.config_id].cfg;
    const int bk = split_box_k(c);
    cudaError_t e;
    if ((e = tc_set_partial(st, st.partial)) != cudaSuccess) return e;
    if ((e = encode_kmajor(st.tmap_a_hi, st.a_hi, M, st.kp, kBM)) != cudaSuccess) return e;
    if ((e = encode_kmajor(st.tmap_a_lo, st.a_lo, M, st.kp, kBM, bk)) != cudaSuccess) return e;
    // a CTA of a pair loads half of the tile's columns of the split B
    const int64_t b_rows = c.bm == 2 * kBM ? c.bn / 2 : c.bn;
    if ((e = encode_kmajor(st.tmap_b_hi, st.b_hi, N, st.kp, b_rows, bk)) != cudaSuccess) return e;
    if ((e = encode_kmajor(st.tmap_b_lo, st.b_lo, N, st.kp, b_rows, bk)) != cudaSuccess) return e;
    return cudaSuccess;
}

namespace {

// How one run goes for the plan's configuration and these operand addresses.
struct Route {
    int id;          // configuration whose main kernel runs
    bool in_kernel;  // the fused kernel (both operands, or A with split B)
    bool raw_a;      // hi of A read from A
    bool pre_a;      // the pre-pass splits A (only lo with raw_a)
    bool pre_b;      // the pre-pass splits B
    bool tmem_a;     // A read from A by the kernel's loader warps into tensor memory
    bool pair;       // a CTA-pair plan whose kernel can take these operands
};

Route route(const TcPlanState& st, const float* A, const float* B)
{
    const TcConfig& c = kTc[st.config_id].cfg;
    const bool a_ok = reinterpret_cast<uintptr_t>(A) % 16 == 0;
    const bool b_ok = reinterpret_cast<uintptr_t>(B) % 16 == 0;
    Route r{};
    r.id = st.config_id;
    r.in_kernel = (c.split == kSplitInKernel && a_ok && b_ok) || (c.split == kSplitHybrid && a_ok);
    r.raw_a = c.split == kSplitRawA && a_ok;
    r.tmem_a = c.split == kSplitTmemA && a_ok;
    r.pre_a = !r.in_kernel && !r.tmem_a;
    r.pre_b = !r.in_kernel || c.split == kSplitHybrid;
    // a misaligned base pointer: the pre-pass form of the same tile width
    if (!r.in_kernel && !r.raw_a && !r.tmem_a && c.split != kSplitPrepass) r.id = st.fallback_config_id;
    r.pair = c.bm == 2 * kBM && (r.in_kernel || r.raw_a || r.tmem_a);
    return r;
}

// The TMA-store map over C, re-encoded when C moves; C's base must be 16-byte
// aligned and ldc and N multiples of 4, else the kernels store C directly.
// (N: a store clipped at the right edge of C was measured to write the whole
// 16-byte chunk holding the last column, i.e. into ldc's padding.)
void prepare_c_map(const TcPlanState& st, float* C, int64_t M, int64_t N, int64_t ldc)
{
    if (reinterpret_cast<uintptr_t>(C) % 16 != 0 || ldc % 4 != 0 || N % 4 != 0) {
        st.c_tma = 0;
        return;
    }
    if (C != st.c_ptr || !st.c_tma) {
        st.c_tma = encode_store_map(st.tmap_c, C, M, N, ldc) == cudaSuccess ? 1 : 0;
        st.c_ptr = C;
    }
}

TcArgs make_args(const TcPlanState& st, int64_t M, int64_t N, float* C, int64_t ldc, int* status)
{
    TcArgs a{};
    a.M = M; a.N = N; a.ldc = ldc; a.C = C; a.partial = st.partial;
    a.status = status;
    a.timeout = st.timeout_cycles > 0 ? st.timeout_cycles : kDefaultTimeout;
    a.tiles_m = st.tiles_m;
    a.tiles_n = st.tiles_n;
    a.num_kb = (int)(st.kp / kBK);
    a.dp_tiles = st.dp_tiles;
    a.split_tiles = st.split_tiles;
    a.splits = st.splits;
    a.kb_per_split = st.kb_per_split;
    a.terms = st.terms;
    a.withhold = st.withhold_stage;
    a.group = st.tile_group > 0 ? st.tile_group : 8;
    a.cluster = st.cluster;
    a.fixup = st.fixup;
    a.gridsum = st.gridsum;
    a.sem = st.sem;
    prepare_c_map(st, C, M, N, ldc);
    a.c_tma = st.c_tma;
    return a;
}

// The operand pre-pass: the A part (rows of this state, only lo with raw_a)
// and/or the B part, one launch.
cudaError_t prepass(const TcPlanState& st, int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                    const float* B, int64_t ldb, bool do_a, bool a_lo_only, bool do_b, cudaStream_t s)
{
    const int vec_a = (lda % 4 == 0) && (reinterpret_cast<uintptr_t>(A) % 16 == 0);
    const int vec_b = (ldb % 4 == 0) && (reinterpret_cast<uintptr_t>(B) % 16 == 0);
    const int a_blocks = do_a ? grid_cap(M * (st.kp / 4), st.num_sms) : 0;
    const int64_t b_blocks = do_b ? (st.kp / kSplitBK) * ((N + kSplitBN - 1) / kSplitBN) : 0;
    if (a_blocks + b_blocks == 0) return cudaSuccess;
    split_operands_kernel<<<(unsigned)(a_blocks + b_blocks), 256, 0, s>>>(
        A, M, K, lda, vec_a, B, N, ldb, vec_b, st.kp, reinterpret_cast<float4*>(st.a_hi),
        reinterpret_cast<float4*>(st.a_lo), st.b_hi, st.b_lo, a_blocks, a_lo_only ? 1 : 0);
    return cudaGetLastError();
}

// The GEMM kernel of the route, then the fixed-order sum of split tiles'
// K-slices over all SMs.  (Summing in the CTA that finishes a tile's last
// slice was measured slower: one CTA's four epilogue warps are latency-bound
// on the slices' L2 reads.)
cudaError_t main_and_reduce(const TcPlanState& st, const Route& r, const TcArgs& a, cudaEvent_t* ev,
                            cudaStream_t s)
{
    const TcConfig& c = kTc[st.config_id].cfg;
    if (a.cluster > 1 && !kTc[r.id].cluster_ok && c.bm != 2 * kBM) return cudaErrorInvalidValue;
    if (a.fixup && !kTc[r.id].fixup_ok) return cudaErrorInvalidValue;
    cudaError_t e;
    if (c.bm == 2 * kBM && r.tmem_a) {
        e = tc_pair_tmem_main(st, a, *reinterpret_cast<const CUtensorMap*>(st.tmap_a_raw),
                              *reinterpret_cast<const CUtensorMap*>(st.tmap_b_hi),
                              *reinterpret_cast<const CUtensorMap*>(st.tmap_b_lo), s);
    } else if (c.bm == 2 * kBM) {
        e = tc_pair_main(c.bn, c.bk, c.split, st, a,
                         *reinterpret_cast<const CUtensorMap*>(st.tmap_a_raw),
                         *reinterpret_cast<const CUtensorMap*>(st.tmap_b_raw),
                         *reinterpret_cast<const CUtensorMap*>(st.tmap_b_hi),
                         *reinterpret_cast<const CUtensorMap*>(st.tmap_b_lo),
                         *reinterpret_cast<const CUtensorMap*>(st.tmap_a_lo), s);
    } else if (r.in_kernel) {
        e = tc_fused_main(c.bn, c.bk, c.split == kSplitHybrid, st, a,
                          *reinterpret_cast<const CUtensorMap*>(st.tmap_a_raw),
                          *reinterpret_cast<const CUtensorMap*>(st.tmap_b_raw),
                          *reinterpret_cast<const CUtensorMap*>(st.tmap_b_hi),
                          *reinterpret_cast<const CUtensorMap*>(st.tmap_b_lo), s);
    } else {
        e = kTc[r.id].main(st, a, r.raw_a ? st.tmap_a_raw : st.tmap_a_hi, s);
    }
    if (e != cudaSuccess) return e;
    if (ev) cudaEventRecord(ev[2], s);
    if (st.split_tiles > 0 && a.cluster <= 1 && !a.fixup && !a.gridsum) e = kTc[r.id].reduce(st, a, s);
    if (ev) cudaEventRecord(ev[3], s);
    return e;
}

}  // namespace

cudaError_t tc_launch(const TcPlanState& st, int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                      const float* B, int64_t ldb, float* C, int64_t ldc, int* status, cudaStream_t s,
                      cudaEvent_t* ev)
{
    const TcConfig& c = kTc[st.config_id].cfg;
    const Route r = route(st, A, B);
    if (c.bm == 2 * kBM && !r.pair) {
        // A CTA-pair plan with a base pointer the TMA cannot take: the one-CTA
        // pre-pass form of the same tile width, its own work decomposition,
        // the same scratch (the partial buffer holds either).
        TcPlanState fb = st;
        fb.config_id = st.fallback_config_id;
        tc_configure(fb, M, N, K, st.split_request);
        // the split operands' maps with the one-CTA tile's rows and 32-k boxes
        const int64_t bn = kTc[fb.config_id].cfg.bn;
        cudaError_t e;
        if ((e = encode_kmajor(fb.tmap_a_lo, fb.a_lo, M, fb.kp, kBM)) != cudaSuccess) return e;
        if ((e = encode_kmajor(fb.tmap_b_hi, fb.b_hi, N, fb.kp, bn)) != cudaSuccess) return e;
        if ((e = encode_kmajor(fb.tmap_b_lo, fb.b_lo, N, fb.kp, bn)) != cudaSuccess) return e;
        return tc_launch(fb, M, N, K, A, lda, B, ldb, C, ldc, status, s, ev);
    }
    cudaError_t e = cudaSuccess;
    if (ev) cudaEventRecord(ev[0], s);
    // Tensor maps over the caller's raw operands, re-encoded when they move.
    if ((r.raw_a || r.tmem_a || r.in_kernel) && A != st.raw_a) {
        if ((e = encode_raw_a(st.tmap_a_raw, A, M, K, lda, c.bk)) != cudaSuccess) return e;
        st.raw_a = A;
    }
    if (r.in_kernel && c.split == kSplitInKernel && B != st.raw_b) {
        if ((e = encode_raw_b(st.tmap_b_raw, B, K, N, ldb, c.bk)) != cudaSuccess) return e;
        st.raw_b = B;
    }
    // 1. The pre-pass into the plan's scratch (what the route needs of it).
    if ((e = prepass(st, M, N, K, A, lda, B, ldb, r.pre_a, r.raw_a, r.pre_b, s)) != cudaSuccess) return e;
    if (ev) cudaEventRecord(ev[1], s);
    // 2. The pipelined tensor-core GEMM and 3. the split tiles' reduction.
    return main_and_reduce(st, r, make_args(st, M, N, C, ldc, status), ev, s);
}

cudaError_t tc_panel_prepare(const TcPlanState& full, int64_t r0, int64_t mp, int64_t N, int64_t K,
                             const float* A, int64_t lda, const float* B, int64_t ldb, TcPlanState& out)
{
    const TcConfig& c = kTc[full.config_id].cfg;
    out = full;
    tc_configure(out, mp, N, K, full.split_request);
    out.partial = nullptr;
    out.sem = nullptr;
    out.c_ptr = nullptr;
    out.c_tma = 0;
    out.a_hi = full.a_hi + r0 * full.kp;
    out.a_lo = full.a_lo + r0 * full.kp;
    cudaError_t e;
    if ((e = encode_kmajor(out.tmap_a_hi, out.a_hi, mp, out.kp, kBM)) != cudaSuccess) return e;
    if ((e = encode_kmajor(out.tmap_a_lo, out.a_lo, mp, out.kp, kBM, split_box_k(c))) != cudaSuccess) return e;
    const Route r = route(out, A + r0 * lda, B);
    if (r.raw_a || r.tmem_a || r.in_kernel) {
        if ((e = encode_raw_a(out.tmap_a_raw, A + r0 * lda, mp, K, lda, c.bk)) != cudaSuccess) return e;
        out.raw_a = A + r0 * lda;
    }
    if (r.in_kernel && c.split == kSplitInKernel) {
        if ((e = encode_raw_b(out.tmap_b_raw, B, K, N, ldb, c.bk)) != cudaSuccess) return e;
        out.raw_b = B;
    }
    return cudaSuccess;
}

cudaError_t tc_block_prepare(const TcPlanState& full, int64_t r0, int64_t mp, int64_t c0, int64_t nq, int64_t K,
                             const float* A, int64_t lda, const float* B, int64_t ldb, TcPlanState& out)
{
    cudaError_t e = tc_panel_prepare(full, r0, mp, nq, K, A, lda, B + c0, ldb, out);
    if (e != cudaSuccess) return e;
    // the block's rows of the split B (B transposed: one row per column of B)
    const TcConfig& c = kTc[full.config_id].cfg;
    out.b_hi = full.b_hi + c0 * full.kp;
    out.b_lo = full.b_lo + c0 * full.kp;
    const int64_t b_rows = c.bm == 2 * kBM ? c.bn / 2 : c.bn;
    if ((e = encode_kmajor(out.tmap_b_hi, out.b_hi, nq, out.kp, b_rows, split_box_k(c))) != cudaSuccess) return e;
    return encode_kmajor(out.tmap_b_lo, out.b_lo, nq, out.kp, b_rows, split_box_k(c));
}

cudaError_t tc_split_b(const TcPlanState& full, int64_t N, int64_t K, const float* A, const float* B,
                       int64_t ldb, cudaStream_t s)
{
    const Route r = route(full, A, B);
    return r.pre_b ? prepass(full, 0, N, K, A, 1, B, ldb, false, false, true, s) : cudaSuccess;
}

cudaError_t tc_panel_run(const TcPlanState& panel, int64_t mp, int64_t N, int64_t K, const float* A_panel,
                         int64_t lda, const float* B, int64_t ldb, float* C_panel, int64_t ldc, int* status,
                         cudaStream_t s, bool pre_a)
{
    const Route r = route(panel, A_panel, B);
    // the panels' operands are the plan's own device buffers, 16-byte aligned
    if (kTc[panel.config_id].cfg.bm == 2 * kBM && !r.pair) return cudaErrorInvalidValue;
    cudaError_t e = prepass(panel, mp, N, K, A_panel, lda, B, ldb, r.pre_a && pre_a, r.raw_a, false, s);
    if (e != cudaSuccess) return e;
    return main_and_reduce(panel, r, make_args(panel, mp, N, C_panel, ldc, status), nullptr, s);
}

}  // namespace gemm_f32
