// C-ABI of the library: plans, the per-shape dispatcher, runs, status codes.
//
// The dispatcher follows the pages' standing lesson that no single kernel is
// fastest ("Double Buffering" technique page, last paragraph; "Case Study: The
// Double-Buffered GEMM", first paragraph): it picks the kernel, its tile, the
// stage count and split-K per problem shape, from a table of timings measured on
// GB300 (dispatch_table.inc) with a rule for shapes the table does not cover.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "internal.h"

using namespace gemm_f32;

namespace {

enum PlanKind : int { kNoop = 0, kZeroFill = 1, kSimt = 2, kTc = 3, kRows = 4, kCols = 5 };
// The short-M and short-N kernels (rows.cu).
constexpr int kVariantRows = GEMM_F32_VARIANT_SHORT_M;
constexpr int kVariantCols = GEMM_F32_VARIANT_SHORT_N;

// Smallest K the tensor-core path accepts (accuracy of the 3xTF32 split):
// 16 with the round-to-nearest split of the pre-pass, 32 with the truncating
// split of the in-kernel path (each product's error is then up to 2^-19|a||b|).
constexpr int64_t kTcMinK = 16;
constexpr int64_t kTcFusedMinK = 32;

struct DispatchChoice {
    int variant;   // GEMM_F32_VARIANT_SIMT / _TCGEN05
    int tile_m, tile_n, stages, split_k;
    int fused;     // TC: where the split happens (kSplitPrepass .. kSplitTmemA)
    int group;     // TC: tile-rows per raster group (0 = default)
    int tile_k;    // SIMT: K-tile depth; TC: k per stage, 32 or 16 (0 = compiled default)
    int k_slices;  // SIMT: K-slice groups inside the CTA (0 = 1)
    int reduce;    // TC: how split tiles' K-slices are summed (the split_reduce option; 0 = kernel)
};

#include "dispatch_table.inc"

}  // namespace

struct gemm_f32_plan_s {
    int64_t M = 0, N = 0, K = 0, lda = 0, ldb = 0, ldc = 0;
    gemm_f32_opts opts{};
    int device = -1;
    int kind = kNoop;
    int num_sms = 0;
    // SIMT path (batch > 1: strided batch of independent products)
    int64_t batch = 1, stride_a = 0, stride_b = 0, stride_c = 0;
    int simt_id = -1;
    int split_k = 1;
    int64_t k_chunk = 0;
    float* partial = nullptr;
    int64_t ldp = 0;
    // tensor-core path
    TcPlanState tc;
    // scratch: one device allocation carved into the buffers above
    void* ws = nullptr;
    size_t ws_bytes = 0;
    int* d_status = nullptr;
    // device staging for gemm_f32_run_host (allocated on first use)
    float* hA = nullptr;
    float* hB = nullptr;
    float* hC = nullptr;
    // two internal streams so the copies of gemm_f32_run_host use two copy engines
    cudaStream_t xs[2] = {nullptr, nullptr};
    cudaEvent_t xev[3] = {nullptr, nullptr, nullptr};
    // row panels of the pipelined gemm_f32_run_host (tensor-core plans): each
    // panel's state and first row, their partial-tile scratch, and one event
    // per landed operand (B, then every A panel) and per finished C panel
    std::vector<TcPlanState> panels;
    std::vector<int64_t> panel_r0;
    // column blocks of the first row panel (host_col_blocks): state, first
    // column; one event per landed B block and per finished C block
    std::vector<TcPlanState> blocks;
    std::vector<int64_t> block_c0;
    int64_t block_width = 0;
    // the last row panel as two column halves (with first-panel blocks, when
    // each half holds a wave of tiles): state, first column; one event per
    // finished half
    std::vector<TcPlanState> tail;
    std::vector<int64_t> tail_c0;
    float* panel_partial = nullptr;
    int* panel_sem = nullptr;
    size_t panel_sem_bytes = 0;
    int panel_count = 0;
    std::vector<cudaEvent_t> pev;
    char desc[256] = {0};
    // tracing: 4 events per recorded run
    std::vector<cudaEvent_t> trace_ev;
    int trace_cap = 0;
    int trace_n = 0;
};

namespace {

gemm_f32_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return GEMM_F32_OK;
    if (e == cudaErrorMemoryAllocation) return GEMM_F32_ERR_OOM;
    return GEMM_F32_ERR_CUDA;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

gemm_f32_status validate_dims(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                              int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0) return GEMM_F32_ERR_INVALID_ARG;
    if (lda < 1 || ldb < 1 || ldc < 1) return GEMM_F32_ERR_INVALID_ARG;
    if (M > 0 && K > 0 && lda < K) return GEMM_F32_ERR_INVALID_ARG;
    if (K > 0 && N > 0 && ldb < N) return GEMM_F32_ERR_INVALID_ARG;
    if (M > 0 && N > 0 && ldc < N) return GEMM_F32_ERR_INVALID_ARG;
    // Keep every index comfortably inside int64 and the grid limits.
    const int64_t lim = int64_t(1) << 31;
    if (M >= lim || N >= lim || K >= lim || lda >= lim || ldb >= lim || ldc >= lim)
        return GEMM_F32_ERR_INVALID_ARG;
    return GEMM_F32_OK;
}

// The options struct as the header lays it out (a binding that mirrors it,
// such as the package's ctypes one, depends on this size).
static_assert(sizeof(gemm_f32_opts) == 72, "gemm_f32_opts layout");

gemm_f32_status validate_opts(const gemm_f32_opts& o)
{
    if (o.variant < 0 || o.variant > GEMM_F32_VARIANT_SHORT_N) return GEMM_F32_ERR_INVALID_ARG;
    if (o.tile_m < 0 || o.tile_n < 0 || o.stages < 0 || o.split_k < 0 || o.split_k > 64)
        return GEMM_F32_ERR_INVALID_ARG;
    if (!(o.tf32_terms == 0 || o.tf32_terms == 1 || o.tf32_terms == 3)) return GEMM_F32_ERR_INVALID_ARG;
    if (o.wait_timeout_cycles < 0 || o.debug_withhold_stage < 0) return GEMM_F32_ERR_INVALID_ARG;
    if (o.separate_syncs != 0 && o.separate_syncs != 1) return GEMM_F32_ERR_INVALID_ARG;
    if (o.operand_split < 0 || o.operand_split > 5) return GEMM_F32_ERR_INVALID_ARG;
    if (o.tile_group < 0 || o.tile_group > 64) return GEMM_F32_ERR_INVALID_ARG;
    if (o.tile_k < 0) return GEMM_F32_ERR_INVALID_ARG;
    if (o.host_panels < 0 || o.host_panels > 64) return GEMM_F32_ERR_INVALID_ARG;
    if (o.split_reduce < 0 || o.split_reduce > 4) return GEMM_F32_ERR_INVALID_ARG;
    if (!(o.k_slices == 0 || o.k_slices == 1 || o.k_slices == 2 || o.k_slices == 4)) return GEMM_F32_ERR_INVALID_ARG;
    if (o.host_col_blocks < 0 || o.host_col_blocks > 16) return GEMM_F32_ERR_INVALID_ARG;
    if (o.simt_fragments != 0 && o.simt_fragments != 1) return GEMM_F32_ERR_INVALID_ARG;
    return GEMM_F32_OK;
}

// Pick a split-K factor so that tiles*split roughly fills the SMs once, with at
// least `min_k_per_split` of K per split.
int auto_split(int64_t tiles, int64_t K, int64_t min_k_per_split, int sms)
{
    if (tiles >= sms / 2) return 1;
    int64_t s = sms / (tiles > 0 ? tiles : 1);
    const int64_t kmax = K / min_k_per_split;
    if (s > kmax) s = kmax;
    if (s > 16) s = 16;
    return s < 1 ? 1 : (int)s;
}

// The rule for tensor-core plans outside the table (checked against the best
// forced plan on 31 shapes the table does not list: squares 768-6144,
// rectangles, skinny and ragged shapes, leading dimensions that are not
// multiples of 4; the sweep is tune.py --rule-sweep):
//   * A's rows not 16-byte aligned (lda not a multiple of 4) or K < 32: only
//     the full pre-pass form can run: 128x256 tiles for big products, 128x128
//     below, a K-split when the tiles fill under half the SMs.
//   * both M and N at least 1000: 256x256 tiles on CTA pairs (one
//     tcgen05.mma across two SMs halves each CTA's B traffic).  Products of
//     2^33 multiply-adds and more read lo of A and B pre-split (no conversion
//     inside the kernel, both CTAs' copies completing on one barrier; 2560^3
//     123 vs 137 us, 4096x1024x4096 138 vs 152 us against splitting in the
//     kernel, 2048^3 a tie); the smaller ones split both operands in the
//     kernel (B by the pre-pass when its rows are not 16-byte aligned), where
//     the pre-pass launch costs more than the conversion it saves; a K-split
//     so that the pairs fill the machine.
//   * otherwise (skinny, or under 1000 on a side): 128x128 tiles on one CTA,
//     operands split in the kernel (B by the pre-pass when its rows are not
//     aligned), K-split to fill the SMs (8192x256x1024 28 vs 40 us,
//     128x4096x4096 30 vs 73 us, 768^3 11.4 vs 15.8 us against the pre-pass
//     form).
DispatchChoice choose_tc(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int sms)
{
    DispatchChoice c{};
    c.variant = GEMM_F32_VARIANT_TCGEN05;
    const double macs = double(M) * double(N) * double(K);
    if (lda % 4 != 0 || K < kTcFusedMinK) {
        c.tile_m = 128;
        c.tile_n = (N >= 2048 && M >= 2048) ? 256 : 128;
        c.fused = kSplitPrepass;
        const int64_t tiles = ((M + 127) / 128) * ((N + c.tile_n - 1) / c.tile_n);
        c.split_k = tiles >= sms / 2 ? 0 : auto_split(tiles, K, 256, sms);
        return c;
    }
    const int b_split = ldb % 4 == 0 ? kSplitInKernel : kSplitHybrid;
    if (M >= 1000 && N >= 1000) {
        c.tile_m = 256;
        c.tile_n = 256;
        c.tile_k = 32;
        c.fused = macs >= 8589934592.0 ? kSplitRawA : b_split;
        const int64_t ptiles = ((M + 255) / 256) * ((N + 255) / 256);
        c.split_k = ptiles >= sms / 4 ? 0 : auto_split(ptiles, K, 192, sms / 2);
        return c;
    }
    c.tile_m = 128;
    c.tile_n = 128;
    c.fused = b_split;
    const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
    c.split_k = tiles >= sms / 2 ? 0 : auto_split(tiles, K, 192, sms);
    return c;
}

// The rule for SIMT plans outside the table: 32x32 tiles of 32-deep K-tiles,
// a 3-stage ring, K split across 4 thread groups of the CTA (more warps per
// SM without a second launch), and a K-split across CTAs only when the tiles
// fill under half the SMs and every slice keeps 128 of K (measured against
// the best forced plan: 64^3 2.04 vs 2.81 us, 200x300x100 2.98 vs 5.78 us,
// 33x65x129 3.5 vs 5.3 us for the rule's earlier 32x32 two-stage plans).
DispatchChoice choose_simt(int64_t M, int64_t N, int64_t K, int sms)
{
    DispatchChoice c{};
    c.variant = GEMM_F32_VARIANT_SIMT;
    c.tile_m = c.tile_n = 32;
    c.stages = 3;
    c.tile_k = 32;
    c.k_slices = 4;
    const int64_t tiles = ((M + 31) / 32) * ((N + 31) / 32);
    // A grid of 32x32 tiles just over the SM count puts two CTAs on a few SMs,
    // which then take twice as long: 32x16 tiles put two on nearly every SM
    // instead (513x257x129 4.65 vs 5.13 us; 512x257x129, 144 tiles, stays at
    // 3.69 with 32x32).  Grids of a few tiles gain from the extra CTAs too
    // (128^3 2.66 vs 2.76 us, 127x193x61 2.12 vs 2.37).
    if ((tiles > sms && tiles <= sms + sms / 4) || tiles <= sms / 8) c.tile_n = 16;
    const int64_t ctas = ((M + 31) / 32) * ((N + c.tile_n - 1) / c.tile_n);
    c.split_k = ctas >= sms / 2 ? 1 : auto_split(ctas, K, 128, sms);
    // Many output tiles over a short K (up to 32): storing C and each CTA's
    // setup dominate, and big tiles without K-slices win: 128x64 while they
    // still give every SM a CTA, else 64x64; 16-deep K-tiles, two stages (the
    // 64x64 tiles a single one when K fits it) (8192x8192x16 78 against 269 us with 32x32 sliced tiles,
    // 16384^2 x 16 300 against 1147, 1024^2 x 16 2.9 against 5.2, 640^2 x 24
    // 2.4 against 2.8).
    const int64_t t64 = ((M + 63) / 64) * ((N + 63) / 64);
    if (K <= 32 && t64 >= sms / 2) {
        const int64_t t128 = ((M + 127) / 128) * ((N + 63) / 64);
        c.tile_m = t128 >= sms ? 128 : 64;
        c.tile_n = 64;
        c.tile_k = 16;
        c.stages = c.tile_m == 64 && K <= 16 ? 1 : 2;
        c.k_slices = 1;
        c.split_k = 1;
    }
    return c;
}

DispatchChoice choose(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int sms)
{
    DispatchChoice c{};
    if (table_lookup(M, N, K, c)) return c;
    // A short A (up to 8 rows) against a large B (2^24 elements or more): the
    // product is bound by reading B, which the short-M kernel streams once
    // (1x8192x8192 49 against 112 us on 128-row tensor-core tiles, whose rows
    // are mostly padding; 8x8192x8192 63 against 112).  With 16 rows its
    // registers cap it under the tensor cores (16x8192x8192 123 against 111),
    // and with a small B its blocks' chain of loads is exposed (1x1024x1024
    // 8.4 against 6.1 us on SIMT tiles).
    if (M <= 8 && double(N) * double(K) >= 16777216.0) {
        c.variant = kVariantRows;
        return c;
    }
    // The mirror case, a single column of B against a large A with rows enough
    // for a warp on each: the short-N kernel (8192x1x8192 66 against 103 us on
    // tensor-core tiles, 65536x1x512 30 against 74).  From two columns its
    // loads of B's rows through L1 bound it (8192x4x8192 588 against 111).
    if (N == 1 && M >= 4096 && double(M) * double(K) >= 16777216.0) {
        c.variant = kVariantCols;
        return c;
    }
    // Shapes outside the measured table: tensor cores once the product is big
    // enough to amortise the operand split; SIMT below that.
    const double macs = double(M) * double(N) * double(K);
    if (macs >= 6.0e7 && K >= 32) return choose_tc(M, N, K, lda, ldb, sms);  // K >= kTcMinK with margin
    // a short K on a large product: the pre-pass form of the tensor cores
    // (8192x2048x24 26 against 31 us on SIMT tiles, 3000x5000x20 27 against 29)
    if (macs >= 2.5e8 && K >= 20) return choose_tc(M, N, K, lda, ldb, sms);
    return choose_simt(M, N, K, sms);
}

gemm_f32_status device_check(int* dev, int* sms)
{
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
        cudaGetLastError();
        return GEMM_F32_ERR_UNSUPPORTED;
    }
    if (cudaGetDevice(dev) != cudaSuccess) return GEMM_F32_ERR_CUDA;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev);
    if (major != 10 || minor != 3) return GEMM_F32_ERR_UNSUPPORTED;
    cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev);
    return GEMM_F32_OK;
}

gemm_f32_status make_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                          int64_t ldc, const gemm_f32_opts* opts_in, gemm_f32_plan_t* out)
{
    if (!out) return GEMM_F32_ERR_INVALID_ARG;
    *out = nullptr;
    gemm_f32_status st = validate_dims(M, N, K, lda, ldb, ldc);
    if (st != GEMM_F32_OK) return st;
    gemm_f32_opts o{};
    if (opts_in) o = *opts_in;
    if ((st = validate_opts(o)) != GEMM_F32_OK) return st;

    gemm_f32_plan_s* p = new (std::nothrow) gemm_f32_plan_s();
    if (!p) return GEMM_F32_ERR_OOM;
    p->M = M; p->N = N; p->K = K; p->lda = lda; p->ldb = ldb; p->ldc = ldc;
    p->opts = o;

    if (M == 0 || N == 0) {
        p->kind = kNoop;
        snprintf(p->desc, sizeof p->desc, "noop M=%lld N=%lld K=%lld", (long long)M,
                 (long long)N, (long long)K);
        *out = p;
        return GEMM_F32_OK;
    }
    if ((st = device_check(&p->device, &p->num_sms)) != GEMM_F32_OK) {
        delete p;
        return st;
    }

    size_t status_off = 0, part_off = 0, ahi_off = 0, alo_off = 0, bhi_off = 0, blo_off = 0, sem_off = 0;
    size_t bytes = align256(sizeof(int));
    status_off = 0;

    if (K == 0) {
        p->kind = kZeroFill;
        snprintf(p->desc, sizeof p->desc, "zero-fill M=%lld N=%lld K=0", (long long)M, (long long)N);
    } else {
        DispatchChoice c = choose(M, N, K, lda, ldb, p->num_sms);
        if (o.variant != GEMM_F32_VARIANT_AUTO && o.variant != c.variant) {
            // A forced variant starts from that variant's own rule.
            if (o.variant == kVariantRows || o.variant == kVariantCols) {
                if (o.variant == kVariantRows ? M > kRowsMaxM : N > kColsMaxN) { delete p; return GEMM_F32_ERR_UNSUPPORTED; }
                c = DispatchChoice{};
                c.variant = o.variant;
            } else {
                c = o.variant == GEMM_F32_VARIANT_SIMT ? choose_simt(M, N, K, p->num_sms)
                                                       : choose_tc(M, N, K, lda, ldb, p->num_sms);
            }
        }
        // Options of the SIMT kernel's shape turn the dispatcher's short-M choice
        // into a SIMT plan (a forced short-M variant takes none of them).
        if ((c.variant == kVariantRows || c.variant == kVariantCols) &&
            (o.tile_m || o.tile_n || o.stages || o.split_k || o.k_slices || o.tile_k || o.separate_syncs ||
             o.simt_fragments)) {
            if (o.variant == kVariantRows || o.variant == kVariantCols) { delete p; return GEMM_F32_ERR_UNSUPPORTED; }
            c = choose_simt(M, N, K, p->num_sms);
        }
        // A forced tile or ring replaces the choice, so the table's K-tile depth
        // and tile order (tuned for its own tile) no longer apply.
        if (o.tile_m || o.tile_n || o.stages) c.tile_k = c.group = c.k_slices = 0;
        if (o.tile_m) c.tile_m = o.tile_m;
        if (o.tile_n) c.tile_n = o.tile_n;
        if (o.stages) c.stages = o.stages;
        if (o.split_k) c.split_k = o.split_k;

        if (c.variant == kVariantCols) {
            p->kind = kCols;
            p->split_k = 1;
            snprintf(p->desc, sizeof p->desc, "simt short-n cols=%lld warp-per-row", (long long)N);
        } else if (c.variant == kVariantRows) {
            p->kind = kRows;
            const int64_t chunk = rows_range(N, K, p->num_sms);
            p->split_k = (int)((K + chunk - 1) / chunk);
            p->k_chunk = chunk;
            if (p->split_k > 1) {
                p->ldp = round_up(N, 4);
                part_off = bytes;
                bytes += align256(size_t(p->split_k) * size_t(M) * size_t(p->ldp) * sizeof(float));
            }
            snprintf(p->desc, sizeof p->desc, "simt short-m rows=%lld cols-per-block=256 k-range=%lld split_k=%d",
                     (long long)M, (long long)chunk, p->split_k);
        } else if (c.variant == GEMM_F32_VARIANT_SIMT) {
            p->kind = kSimt;
            const int ksl = o.k_slices ? o.k_slices : c.k_slices ? c.k_slices : 1;
            p->simt_id = simt_find_config(c.tile_m, c.tile_n, c.stages, o.separate_syncs != 0,
                                          o.tile_k ? o.tile_k : c.tile_k, ksl, o.simt_fragments != 0);
            if (p->simt_id < 0) { delete p; return GEMM_F32_ERR_UNSUPPORTED; }
            const int bk = simt_config(p->simt_id).bk;
            int64_t split = c.split_k < 1 ? 1 : c.split_k;
            int64_t chunk = round_up((K + split - 1) / split, bk);
            split = (K + chunk - 1) / chunk;  // no empty splits
            p->split_k = (int)split;
            p->k_chunk = chunk;
            if (split > 1) {
                p->ldp = round_up(N, 4);
                part_off = bytes;
                bytes += align256(size_t(split) * size_t(M) * size_t(p->ldp) * sizeof(float));
            }
            const SimtConfig& sc = simt_config(p->simt_id);
            char ks[24] = "";
            if (sc.ksl > 1) snprintf(ks, sizeof ks, " k_slices=%d", sc.ksl);
            snprintf(p->desc, sizeof p->desc,
                     "simt tile=%dx%dx%d thread=%dx%d stages=%d%s%s%s split_k=%d", sc.bm, sc.bn, sc.bk,
                     sc.tm, sc.tn, sc.stages, sc.sep ? " separate-syncs" : "", ks,
                     sc.shfl ? " shuffle-fragments" : "", p->split_k);
        } else {
            // The two-piece TF32 split keeps 22 of FP32's 24 significand bits, so
            // each product carries an error up to about 3*2^-22*|a||b|; against the
            // bound 2*K*2^-24*sum|a||b| that fits only once K is about 10 or more.
            if (K < kTcMinK) { delete p; return GEMM_F32_ERR_UNSUPPORTED; }
            p->kind = kTc;
            TcPlanState& t = p->tc;
            // operand_split: 1 pre-pass, 2 in the kernel, 3 hybrid (A in the kernel,
            // B by the pre-pass), 4 hi of A read from A, 5 A split by the pairs'
            // loader warps into tensor memory; 0 = the dispatcher's choice.
            // A forced ring depth exists only in the pre-pass form (the other
            // forms have one depth per tile width), so it selects that form.
            // Half-size (16-k) stages exist only in the in-kernel form, so a
            // forced tile_k of 16 selects that form.
            // tile_m 256: a pair of CTAs per 256-row tile (one tcgen05.mma
            // across both), operands split in the kernel only.
            // operand_split 3 (B by the pre-pass) asks for the pairs' hybrid form,
            // 4 (lo of A and B by the pre-pass) for their form without converters,
            // 5 for their form with A in tensor memory
            bool pair = c.tile_m == 256;
            const int pair_split = o.operand_split == 5   ? kSplitTmemA
                                   : o.operand_split == 4 ? kSplitRawA
                                   : o.operand_split == 3 ? kSplitHybrid
                                   : o.operand_split      ? kSplitInKernel
                                   : (c.fused == kSplitHybrid || c.fused == kSplitRawA || c.fused == kSplitTmemA)
                                         ? c.fused
                                         : kSplitInKernel;
            if (pair && (o.operand_split == 1 || o.stages ||
                         o.separate_syncs || o.split_reduce == 3 || K < kTcFusedMinK || lda % 4 != 0 ||
                         (pair_split == kSplitInKernel && ldb % 4 != 0))) {
                // forced: refused; the dispatcher's choice: the one-CTA kernel
                if (o.tile_m == 256) { delete p; return GEMM_F32_ERR_UNSUPPORTED; }
                pair = false;
                c.tile_m = 128;
                c.fused = kSplitPrepass;
                c.tile_k = 0;
            }
            if (pair) {
                const int pbk = o.tile_k ? o.tile_k : c.tile_k;
                t.config_id = tc_find_pair_config(c.tile_n, pbk, pair_split);
                if (t.config_id < 0) { delete p; return GEMM_F32_ERR_UNSUPPORTED; }
                t.pair_slots = tc_pair_slots(c.tile_n, tc_config(t.config_id).bk, p->num_sms, pair_split);
                if (t.pair_slots < 1) { delete p; return GEMM_F32_ERR_UNSUPPORTED; }
                t.fallback_config_id = tc_find_config(c.tile_n, 0, false, kSplitPrepass);
            } else {
                int where = o.operand_split ? o.operand_split - 1
                            : o.stages      ? kSplitPrepass
                            : o.tile_k == 16 ? kSplitInKernel
                                             : c.fused;
                const int tc_bk = where == kSplitInKernel ? (o.tile_k ? o.tile_k : c.tile_k) : 0;
                const bool ok = where == kSplitPrepass ||
                                (K >= kTcFusedMinK && lda % 4 == 0 && (where != kSplitInKernel || ldb % 4 == 0) &&
                                 !o.separate_syncs && tc_find_config(c.tile_n, 0, false, where, tc_bk) >= 0);
                if (!ok) {
                    if (o.operand_split || o.tile_k == 16) { delete p; return GEMM_F32_ERR_UNSUPPORTED; }
                    where = kSplitPrepass;
                }
                if (o.tile_k && where != kSplitInKernel && o.tile_k != 32) { delete p; return GEMM_F32_ERR_UNSUPPORTED; }
                t.config_id = tc_find_config(c.tile_n, where != kSplitPrepass ? 0 : c.stages, o.separate_syncs != 0,
                                             where, where == kSplitInKernel ? tc_bk : 0);
                if (c.tile_m != 128 || t.config_id < 0) { delete p; return GEMM_F32_ERR_UNSUPPORTED; }
                if (where != kSplitPrepass) t.fallback_config_id = tc_find_config(c.tile_n, 0, false, kSplitPrepass);
            }
            const TcConfig& tcfg = tc_config(t.config_id);
            t.terms = o.tf32_terms ? o.tf32_terms : 3;
            t.num_sms = p->num_sms;
            t.timeout_cycles = o.wait_timeout_cycles;
            t.withhold_stage = o.debug_withhold_stage;
            t.tile_group = o.tile_group ? o.tile_group : c.group;
            // the table's K-slice sum goes with its own split
            t.cluster_mode = o.split_reduce ? o.split_reduce : o.split_k ? 0 : c.reduce;
            tc_configure(t, M, N, K, c.split_k);
            if ((o.split_reduce == 2 && t.cluster == 0) || (o.split_reduce == 3 && t.fixup == 0) ||
                (o.split_reduce == 4 && t.gridsum == 0)) {
                delete p;
                return GEMM_F32_ERR_UNSUPPORTED;
            }
            if (pair) {
                // a run with operands the TMA cannot take falls back to the
                // one-CTA pre-pass form: the partial buffer holds either's slices
                TcPlanState fb = t;
                fb.config_id = t.fallback_config_id;
                tc_configure(fb, M, N, K, c.split_k);
                if (fb.partial_bytes > t.partial_bytes) t.partial_bytes = fb.partial_bytes;
            }
            ahi_off = bytes; bytes += align256(size_t(M) * size_t(t.kp) * sizeof(float));
            alo_off = bytes; bytes += align256(size_t(M) * size_t(t.kp) * sizeof(float));
            bhi_off = bytes; bytes += align256(size_t(N) * size_t(t.kp) * sizeof(float));
            blo_off = bytes; bytes += align256(size_t(N) * size_t(t.kp) * sizeof(float));
            if (t.partial_bytes) {
                part_off = bytes;
                bytes += align256(t.partial_bytes);
            }
            if (t.sem_bytes) {
                sem_off = bytes;
                bytes += align256(t.sem_bytes);
            }
            if (pair)
                snprintf(p->desc, sizeof p->desc,
                         "tcgen05 3xtf32 %s cta-pair terms=%d tile=%dx%dx%d stages=%d pairs=%d "
                         "whole=%d split=%dx%d%s resident=%d group=%d kp=%lld",
                         tcfg.split == kSplitHybrid ? "hybrid-split"
                         : tcfg.split == kSplitRawA ? "raw-a-split"
                         : tcfg.split == kSplitTmemA ? "tmem-a-split" : "in-kernel-split", t.terms, tcfg.bm, tcfg.bn, tcfg.bk, tcfg.stages, t.tiles_m / 2 * t.tiles_n, t.dp_tiles,
                         t.split_tiles, t.splits, t.cluster ? " cluster-sum" : t.gridsum ? " grid-sum" : "",
                         t.pair_slots,
                         t.tile_group > 0 ? t.tile_group : 8,
                         (long long)t.kp);
            else
                snprintf(p->desc, sizeof p->desc,
                         "tcgen05 3xtf32%s terms=%d tile=%dx%dx%d stages=%d%s tiles=%d whole=%d split=%dx%d%s "
                         "group=%d kp=%lld",
                         tcfg.split == kSplitInKernel ? " in-kernel-split"
                         : tcfg.split == kSplitHybrid ? " hybrid-split"
                         : tcfg.split == kSplitRawA ? " raw-a-split" : "",
                         t.terms, tcfg.bm, tcfg.bn, tcfg.bk, tcfg.stages,
                         tcfg.sep ? " separate-syncs" : "",
                         t.tiles_m * t.tiles_n, t.dp_tiles,
                         t.split_tiles, t.splits, t.cluster ? " cluster-sum" : t.fixup ? " last-arriver-sum" : "",
                         t.tile_group > 0 ? t.tile_group : 8, (long long)t.kp);
        }
    }

    cudaError_t e = cudaMalloc(&p->ws, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return from_cuda(e);
    }
    p->ws_bytes = bytes;
    char* base = static_cast<char*>(p->ws);
    p->d_status = reinterpret_cast<int*>(base + status_off);
    e = cudaMemset(p->d_status, 0, sizeof(int));
    if ((p->kind == kSimt || p->kind == kRows) && p->split_k > 1) p->partial = reinterpret_cast<float*>(base + part_off);
    if (p->kind == kTc) {
        TcPlanState& t = p->tc;
        t.a_hi = reinterpret_cast<float*>(base + ahi_off);
        t.a_lo = reinterpret_cast<float*>(base + alo_off);
        t.b_hi = reinterpret_cast<float*>(base + bhi_off);
        t.b_lo = reinterpret_cast<float*>(base + blo_off);
        if (t.partial_bytes) t.partial = reinterpret_cast<float*>(base + part_off);
        if (t.sem_bytes) {
            t.sem = reinterpret_cast<int*>(base + sem_off);
            if (e == cudaSuccess) e = cudaMemset(t.sem, 0, t.sem_bytes);
        }
        if (e == cudaSuccess) e = tc_prepare(t, M, N, K);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p->ws);
        delete p;
        return from_cuda(e);
    }
    size_t len = strlen(p->desc);
    snprintf(p->desc + len, sizeof p->desc - len, " ws=%zu", p->ws_bytes);
    *out = p;
    return GEMM_F32_OK;
}

// Copy a rows x cols matrix with leading dimension ld (same on both sides):
// one linear copy when the rows are contiguous, a pitched copy otherwise
// (so the destination's padding columns are never written).
cudaError_t copy_rows(float* dst, const float* src, int64_t rows, int64_t cols, int64_t ld,
                      cudaMemcpyKind kind, cudaStream_t s)
{
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    if (ld == cols || rows == 1)
        return cudaMemcpyAsync(dst, src, size_t(rows) * size_t(cols) * sizeof(float), kind, s);
    return cudaMemcpy2DAsync(dst, size_t(ld) * sizeof(float), src, size_t(ld) * sizeof(float),
                             size_t(cols) * sizeof(float), size_t(rows), kind, s);
}

bool current_device_is(int dev)
{
    int d = -1;
    return cudaGetDevice(&d) == cudaSuccess && d == dev;
}

// Column blocks of the first row panel asked for (before rounding to whole
// tiles): the option's count, else 3 from N = 6144 and 2 from N = 2048
// (measured on GB300, pinned host memory at about 200 GB/s each way: 8192^3
// 5.18 ms with 5 panels and 3 blocks against 6.04 ms with 6 panels and none;
// 4096^3 1.08 ms with 3 panels and 2 blocks against 1.12 ms with none, 1.27
// with 4).  For plans whose A is split in the GEMM kernel or reads hi of A
// from A (the blocks share the first panel's pre-split lo of A, made once by
// the first block); the full pre-pass form keeps whole panels.
int host_col_request(const gemm_f32_plan_s* p)
{
    const TcConfig& c = tc_config(p->tc.config_id);
    if (c.split == kSplitPrepass) return 1;
    const int q = p->opts.host_col_blocks;
    // 4 blocks from N = 6144 (8192^3 with its first panel of two shares: 4.38
    // against 4.49 ms with 3), 2 from N = 2048
    return q != 0 ? q : p->N >= 6144 ? 4 : p->N >= 2048 ? 2 : 1;
}

// Row panels of the pipelined host-buffer run: the option's count, else a
// count from the waves of output tiles (measured on GB300 with pinned host
// memory at about 200 GB/s each way: 8192^3, 13 waves, is fastest with 6
// panels, or 5 when the first panel runs in column blocks; 4096^3, 3.4
// waves, with 3); never more panels than tile-rows.  1 = the plain
// copy-run-copy sequence.
int host_panel_count(const gemm_f32_plan_s* p)
{
    if (p->kind != kTc || p->K == 0) return 1;
    int n = p->opts.host_panels;
    if (n == 0) {
        const int64_t waves = int64_t(p->tc.tiles_m) * p->tc.tiles_n / (p->num_sms > 0 ? p->num_sms : 1);
        n = waves >= 8 ? (host_col_request(p) > 1 ? 5 : 6) : waves >= 2 ? 3 : waves >= 1 ? 2 : 1;
    }
    // whole tile rows per panel (two 128-row tiles for a CTA-pair plan)
    const int tile_rows = p->tc.tiles_m / (tc_config(p->tc.config_id).bm / 128);
    if (n > tile_rows) n = tile_rows;
    return n < 1 ? 1 : n;
}

// Width of the first row panel's column blocks (whole tiles), 0 = no blocks
// (fewer than two row panels, or one block).  Without blocks the copy of B,
// 1.3 ms at 8192 x 8192, comes whole before the first GEMM.
int64_t host_col_width(const gemm_f32_plan_s* p, int panels)
{
    const int q = host_col_request(p);
    if (panels < 2 || q <= 1) return 0;
    const int64_t w = round_up((p->N + q - 1) / q, tc_config(p->tc.config_id).bn);
    return w < p->N ? w : 0;
}

void drop_panels(gemm_f32_plan_s* p)
{
    p->panels.clear();
    p->panel_r0.clear();
    p->blocks.clear();
    p->block_c0.clear();
    p->block_width = 0;
    p->tail.clear();
    p->tail_c0.clear();
    p->panel_count = 0;
    if (p->panel_partial) cudaFree(p->panel_partial);
    p->panel_partial = nullptr;
    if (p->panel_sem) cudaFree(p->panel_sem);
    p->panel_sem = nullptr;
    p->panel_sem_bytes = 0;
}

// Panel states for `count` panels of whole 128-row tiles over the staging
// buffers (and the first panel's column blocks of `width` columns, 0 = none),
// their partial-tile scratch and events; kept until the counts change.
cudaError_t make_panels(gemm_f32_plan_s* p, int count, int64_t width)
{
    if (!p->panels.empty() && p->panel_count == count && p->block_width == width) return cudaSuccess;
    drop_panels(p);
    const int64_t bm = tc_config(p->tc.config_id).bm;
    int64_t rows = round_up((p->M + count - 1) / count, bm);
    // With column blocks on a GEMM of many waves (copies shorter than the
    // GEMM), the first panel takes two shares of the tile rows: its blocks'
    // GEMMs then last about as long as the copy of the next block of B, so
    // the GEMM does not wait between them.
    int64_t first = rows;
    const int64_t waves = int64_t(p->tc.tiles_m) * p->tc.tiles_n / (p->num_sms > 0 ? p->num_sms : 1);
    if (width > 0 && count > 2 && waves >= 8) {
        const int64_t tile_rows = (p->M + bm - 1) / bm, share = tile_rows / (count + 1);
        if (share >= 1) {
            rows = share * bm;
            first = (tile_rows - share * (count - 1)) * bm;
        }
    }
    size_t need = 0;
    cudaError_t e = cudaSuccess;
    for (int64_t r0 = 0; r0 < p->M; r0 += r0 == 0 ? first : rows) {
        const int64_t step = r0 == 0 ? first : rows;
        const int64_t mp = p->M - r0 < step ? p->M - r0 : step;
        TcPlanState ps;
        if ((e = tc_panel_prepare(p->tc, r0, mp, p->N, p->K, p->hA, p->lda, p->hB, p->ldb, ps)) != cudaSuccess) {
            drop_panels(p);
            return e;
        }
        if (ps.partial_bytes > need) need = ps.partial_bytes;
        if (ps.sem_bytes > p->panel_sem_bytes) p->panel_sem_bytes = ps.sem_bytes;
        p->panels.push_back(ps);
        p->panel_r0.push_back(r0);
    }
    const int64_t mp0 = p->panels.size() > 1 ? p->panel_r0[1] : p->M;
    for (int64_t c0 = 0; width > 0 && c0 < p->N; c0 += width) {
        TcPlanState bs;
        const int64_t nq = p->N - c0 < width ? p->N - c0 : width;
        if ((e = tc_block_prepare(p->tc, 0, mp0, c0, nq, p->K, p->hA, p->lda, p->hB, p->ldb, bs)) != cudaSuccess) {
            drop_panels(p);
            return e;
        }
        if (bs.partial_bytes > need) need = bs.partial_bytes;
        if (bs.sem_bytes > p->panel_sem_bytes) p->panel_sem_bytes = bs.sem_bytes;
        p->blocks.push_back(bs);
        p->block_c0.push_back(c0);
    }
    // The last panel in two column halves, the first half's C copied back
    // while the second half's GEMM runs: only half a panel of C is left to
    // copy after the last GEMM.  Only where each half keeps every CTA (pair)
    // busy for a wave (8192^3: 0.22 ms of copy after the GEMMs, of 4.4).
    const int64_t bn = tc_config(p->tc.config_id).bn;
    const int64_t half = round_up((p->N + 1) / 2, bn);
    if (width > 0 && count > 2 && half < p->N) {
        const int64_t r0 = p->panel_r0.back(), mp = p->M - r0;
        const int64_t slots = p->tc.pair_slots > 0 ? int64_t(p->tc.pair_slots) : int64_t(p->num_sms);
        const int64_t half_tiles = (mp + bm - 1) / bm * ((p->N - half + bn - 1) / bn);
        if (half_tiles >= slots) {
            for (int64_t c0 = 0; c0 < p->N; c0 += half) {
                TcPlanState ts;
                const int64_t nq = p->N - c0 < half ? p->N - c0 : half;
                if ((e = tc_block_prepare(p->tc, r0, mp, c0, nq, p->K, p->hA, p->lda, p->hB, p->ldb, ts)) !=
                    cudaSuccess) {
                    drop_panels(p);
                    return e;
                }
                if (ts.partial_bytes > need) need = ts.partial_bytes;
                if (ts.sem_bytes > p->panel_sem_bytes) p->panel_sem_bytes = ts.sem_bytes;
                p->tail.push_back(ts);
                p->tail_c0.push_back(c0);
            }
        }
    }
    if (need && (e = cudaMalloc(&p->panel_partial, need)) != cudaSuccess) {
        p->panel_partial = nullptr;
        drop_panels(p);
        return e;
    }
    // the panels run one after another and leave their counters at zero, so
    // they share one zeroed counter buffer
    if (p->panel_sem_bytes) {
        e = cudaMalloc(&p->panel_sem, p->panel_sem_bytes);
        if (e == cudaSuccess) e = cudaMemset(p->panel_sem, 0, p->panel_sem_bytes);
        if (e != cudaSuccess) {
            drop_panels(p);
            return e;
        }
    }
    for (std::vector<TcPlanState>* v : {&p->panels, &p->blocks, &p->tail})
        for (TcPlanState& ps : *v) {
            if (e == cudaSuccess) e = tc_set_partial(ps, p->panel_partial);
            ps.sem = ps.sem_bytes ? p->panel_sem : nullptr;
        }
    if (e != cudaSuccess) {
        drop_panels(p);
        return e;
    }
    while (e == cudaSuccess && p->pev.size() < 1 + 2 * p->panels.size() + 2 * p->blocks.size() + p->tail.size()) {
        cudaEvent_t x = nullptr;
        e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
        if (e == cudaSuccess) p->pev.push_back(x);
    }
    if (e != cudaSuccess) {
        drop_panels(p);
    } else {
        p->panel_count = count;
        p->block_width = width;
    }
    return e;
}

// The panel pipeline.  Stream xs[0] copies B, then every A panel, each
// followed by an event; the caller's stream splits B once and runs each
// panel's pre-pass, GEMM and reduction after its A panel has landed; stream
// xs[1] copies each C panel back once it is done.  So panel i's GEMM overlaps
// the copy of A panel i+1 and of C panel i-1.
//
// With column blocks, the first panel is the blocks instead: xs[0] copies B
// block 0, A panel 0, then the other B blocks (each a pitched copy of its
// columns), then A panels 1..; the caller's stream splits each B block as it
// lands and runs its block of the first panel (rows of panel 0, the block's
// columns), then panels 1.. over the whole of B; xs[1] copies each C block
// and then each C panel back.  The first GEMM waits for one block of B and
// one panel of A instead of all of B.  With the last panel in two column
// halves, each half's C is copied back as soon as its GEMM is done.
cudaError_t run_host_panels(gemm_f32_plan_s* p, const float* A_host, const float* B_host, float* C_host,
                            cudaStream_t s)
{
    const size_t np = p->panels.size(), nb = p->blocks.size(), nt = p->tail.size();
    cudaEvent_t ev_b = p->pev[0];
    const cudaEvent_t* ev_a = &p->pev[1];
    const cudaEvent_t* ev_c = &p->pev[1 + np];
    const cudaEvent_t* ev_bb = &p->pev[1 + 2 * np];
    const cudaEvent_t* ev_cb = &p->pev[1 + 2 * np + nb];
    const cudaEvent_t* ev_ct = &p->pev[1 + 2 * np + 2 * nb];
    auto panel_rows = [&](size_t i) { return (i + 1 < np ? p->panel_r0[i + 1] : p->M) - p->panel_r0[i]; };
    auto block_cols = [&](size_t j) { return (j + 1 < nb ? p->block_c0[j + 1] : p->N) - p->block_c0[j]; };
    auto tail_cols = [&](size_t j) { return (j + 1 < nt ? p->tail_c0[j + 1] : p->N) - p->tail_c0[j]; };
    // the whole panels: all but the first with column blocks, all but the last with column halves
    const size_t first_whole = nb == 0 ? 0 : 1, end_whole = nt == 0 ? np : np - 1;
    // a rows x cols block at column c0 of a matrix with leading dimension ld
    auto copy_block = [](float* dst, const float* src, int64_t rows, int64_t cols, int64_t ld, cudaMemcpyKind kind,
                         cudaStream_t st) -> cudaError_t {
        if (rows <= 0 || cols <= 0) return cudaSuccess;
        return cudaMemcpy2DAsync(dst, size_t(ld) * sizeof(float), src, size_t(ld) * sizeof(float),
                                 size_t(cols) * sizeof(float), size_t(rows), kind, st);
    };
    cudaError_t e;
    // both copy streams start after the caller's earlier work
    if ((e = cudaEventRecord(p->xev[0], s)) != cudaSuccess) return e;
    for (int i = 0; i < 2; ++i)
        if ((e = cudaStreamWaitEvent(p->xs[i], p->xev[0], 0)) != cudaSuccess) return e;
    // host -> device: B (whole, or block 0 with the other blocks after A panel 0), then the A panels
    auto copy_a = [&](size_t i) -> cudaError_t {
        const int64_t r0 = p->panel_r0[i];
        cudaError_t r = copy_rows(p->hA + r0 * p->lda, A_host + r0 * p->lda, panel_rows(i), p->K, p->lda,
                                  cudaMemcpyHostToDevice, p->xs[0]);
        return r == cudaSuccess ? cudaEventRecord(ev_a[i], p->xs[0]) : r;
    };
    if (nb == 0) {
        if ((e = copy_rows(p->hB, B_host, p->K, p->N, p->ldb, cudaMemcpyHostToDevice, p->xs[0])) != cudaSuccess ||
            (e = cudaEventRecord(ev_b, p->xs[0])) != cudaSuccess || (e = copy_a(0)) != cudaSuccess)
            return e;
    } else {
        for (size_t j = 0; j < nb; ++j) {
            const int64_t c0 = p->block_c0[j];
            if ((e = copy_block(p->hB + c0, B_host + c0, p->K, block_cols(j), p->ldb, cudaMemcpyHostToDevice,
                                p->xs[0])) != cudaSuccess ||
                (e = cudaEventRecord(ev_bb[j], p->xs[0])) != cudaSuccess)
                return e;
            if (j == 0 && (e = copy_a(0)) != cudaSuccess) return e;
        }
    }
    for (size_t i = 1; i < np; ++i)
        if ((e = copy_a(i)) != cudaSuccess) return e;
    // compute: the first panel (whole, after B's split, or block by block), then the others
    if (nb == 0) {
        if ((e = cudaStreamWaitEvent(s, ev_b, 0)) != cudaSuccess ||
            (e = tc_split_b(p->tc, p->N, p->K, p->hA, p->hB, p->ldb, s)) != cudaSuccess)
            return e;
    } else {
        for (size_t j = 0; j < nb; ++j) {
            const int64_t c0 = p->block_c0[j];
            if ((e = cudaStreamWaitEvent(s, ev_bb[j], 0)) != cudaSuccess ||
                (e = tc_split_b(p->blocks[j], block_cols(j), p->K, p->hA, p->hB + c0, p->ldb, s)) != cudaSuccess ||
                (j == 0 && (e = cudaStreamWaitEvent(s, ev_a[0], 0)) != cudaSuccess) ||
                (e = tc_panel_run(p->blocks[j], panel_rows(0), block_cols(j), p->K, p->hA, p->lda, p->hB + c0,
                                  p->ldb, p->hC + c0, p->ldc, p->d_status, s, j == 0)) != cudaSuccess ||
                (e = cudaEventRecord(ev_cb[j], s)) != cudaSuccess)
                return e;
        }
    }
    for (size_t i = first_whole; i < end_whole; ++i) {
        const int64_t r0 = p->panel_r0[i];
        if ((e = cudaStreamWaitEvent(s, ev_a[i], 0)) != cudaSuccess ||
            (e = tc_panel_run(p->panels[i], panel_rows(i), p->N, p->K, p->hA + r0 * p->lda, p->lda, p->hB, p->ldb,
                              p->hC + r0 * p->ldc, p->ldc, p->d_status, s)) != cudaSuccess ||
            (e = cudaEventRecord(ev_c[i], s)) != cudaSuccess)
            return e;
    }
    // the last panel's halves: the first makes the panel's pre-split A for both
    if (nt > 0) {
        const int64_t r0 = p->panel_r0[np - 1];
        if ((e = cudaStreamWaitEvent(s, ev_a[np - 1], 0)) != cudaSuccess) return e;
        for (size_t j = 0; j < nt; ++j) {
            const int64_t c0 = p->tail_c0[j];
            if ((e = tc_panel_run(p->tail[j], panel_rows(np - 1), tail_cols(j), p->K, p->hA + r0 * p->lda, p->lda,
                                  p->hB + c0, p->ldb, p->hC + r0 * p->ldc + c0, p->ldc, p->d_status, s,
                                  j == 0)) != cudaSuccess ||
                (e = cudaEventRecord(ev_ct[j], s)) != cudaSuccess)
                return e;
        }
    }
    // device -> host: each C block and C panel when it is done; the caller's stream joins.
    // The C blocks wait for the last B block too: until then the host link's
    // other direction carries B, which the GEMMs are waiting for.
    if (nb > 0 && (e = cudaStreamWaitEvent(p->xs[1], ev_bb[nb - 1], 0)) != cudaSuccess) return e;
    for (size_t j = 0; j < nb; ++j) {
        const int64_t c0 = p->block_c0[j];
        if ((e = cudaStreamWaitEvent(p->xs[1], ev_cb[j], 0)) != cudaSuccess ||
            (e = copy_block(C_host + c0, p->hC + c0, panel_rows(0), block_cols(j), p->ldc, cudaMemcpyDeviceToHost,
                            p->xs[1])) != cudaSuccess)
            return e;
    }
    for (size_t i = first_whole; i < end_whole; ++i) {
        const int64_t r0 = p->panel_r0[i];
        if ((e = cudaStreamWaitEvent(p->xs[1], ev_c[i], 0)) != cudaSuccess ||
            (e = copy_rows(C_host + r0 * p->ldc, p->hC + r0 * p->ldc, panel_rows(i), p->N, p->ldc,
                           cudaMemcpyDeviceToHost, p->xs[1])) != cudaSuccess)
            return e;
    }
    for (size_t j = 0; j < nt; ++j) {
        const int64_t r0 = p->panel_r0[np - 1], c0 = p->tail_c0[j];
        if ((e = cudaStreamWaitEvent(p->xs[1], ev_ct[j], 0)) != cudaSuccess ||
            (e = copy_block(C_host + r0 * p->ldc + c0, p->hC + r0 * p->ldc + c0, panel_rows(np - 1), tail_cols(j),
                            p->ldc, cudaMemcpyDeviceToHost, p->xs[1])) != cudaSuccess)
            return e;
    }
    if ((e = cudaEventRecord(p->xev[2], p->xs[1])) != cudaSuccess) return e;
    return cudaStreamWaitEvent(s, p->xev[2], 0);
}

}  // namespace

extern "C" {

gemm_f32_status gemm_f32_opts_init(gemm_f32_opts* opts)
{
    if (!opts) return GEMM_F32_ERR_INVALID_ARG;
    memset(opts, 0, sizeof *opts);
    return GEMM_F32_OK;
}

gemm_f32_status gemm_f32_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                              int64_t ldc, gemm_f32_plan_t* plan)
{
    return make_plan(M, N, K, lda, ldb, ldc, nullptr, plan);
}

gemm_f32_status gemm_f32_plan_ex(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                 int64_t ldc, const gemm_f32_opts* opts, gemm_f32_plan_t* plan)
{
    return make_plan(M, N, K, lda, ldb, ldc, opts, plan);
}

gemm_f32_status gemm_f32_plan_batched(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                      int64_t ldc, int64_t batch, int64_t stride_a, int64_t stride_b,
                                      int64_t stride_c, const gemm_f32_opts* opts, gemm_f32_plan_t* plan)
{
    if (!plan) return GEMM_F32_ERR_INVALID_ARG;
    *plan = nullptr;
    if (batch < 0 || batch > 65535 || stride_a < 0 || stride_b < 0 || stride_c < 0)
        return GEMM_F32_ERR_INVALID_ARG;
    gemm_f32_status st = validate_dims(M, N, K, lda, ldb, ldc);
    if (st != GEMM_F32_OK) return st;
    if (batch > 1 && M > 0 && N > 0 && stride_c < (M - 1) * ldc + N) return GEMM_F32_ERR_INVALID_ARG;
    gemm_f32_opts o{};
    if (opts) o = *opts;
    if (o.variant != GEMM_F32_VARIANT_AUTO && o.variant != GEMM_F32_VARIANT_SIMT) return GEMM_F32_ERR_UNSUPPORTED;
    if (batch <= 1 || M == 0 || N == 0) {
        // one product (or none): an ordinary plan
        if (batch == 0) return make_plan(0, N, K, lda, ldb, ldc, &o, plan);
        o.variant = o.variant ? o.variant : GEMM_F32_VARIANT_AUTO;
        return make_plan(M, N, K, lda, ldb, ldc, &o, plan);
    }
    // SIMT tile for the per-product shape; no split-K (the batch fills the GPU).
    o.variant = GEMM_F32_VARIANT_SIMT;
    if (!o.tile_m || !o.tile_n) {
        const int64_t d = M > N ? M : N;
        o.tile_m = o.tile_n = d <= 32 ? 32 : d <= 64 ? 64 : 128;
        if (!o.stages) o.stages = d <= 32 ? 1 : 2;
    }
    if (!o.stages) o.stages = 2;
    o.split_k = 1;
    st = make_plan(M, N, K, lda, ldb, ldc, &o, plan);
    if (st != GEMM_F32_OK) return st;
    gemm_f32_plan_s* p = *plan;
    p->batch = batch;
    p->stride_a = stride_a;
    p->stride_b = stride_b;
    p->stride_c = stride_c;
    const size_t len = strlen(p->desc);
    snprintf(p->desc + len, sizeof p->desc - len, " batch=%lld", (long long)batch);
    return GEMM_F32_OK;
}

gemm_f32_status gemm_f32_run(gemm_f32_plan_t p, const float* A, const float* B, float* C,
                             gemm_f32_stream_t stream)
{
    if (!p) return GEMM_F32_ERR_INVALID_ARG;
    if (p->kind == kNoop) return GEMM_F32_OK;
    if (!C || (p->K > 0 && (!A || !B))) return GEMM_F32_ERR_INVALID_ARG;
    if (!current_device_is(p->device)) return GEMM_F32_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    cudaEvent_t* ev = nullptr;
    if (p->trace_n < p->trace_cap) ev = &p->trace_ev[4 * size_t(p->trace_n++)];
    switch (p->kind) {
    case kZeroFill:
        if (ev) { cudaEventRecord(ev[0], s); cudaEventRecord(ev[1], s); }
        for (int64_t z = 0; z < p->batch && e == cudaSuccess; ++z)
            e = zero_fill_launch(C + z * p->stride_c, p->M, p->N, p->ldc, s);
        if (ev) { cudaEventRecord(ev[2], s); cudaEventRecord(ev[3], s); }
        break;
    case kSimt: {
        SimtArgs a{};
        a.M = p->M; a.N = p->N; a.K = p->K;
        a.A = A; a.lda = p->lda; a.B = B; a.ldb = p->ldb; a.C = C; a.ldc = p->ldc;
        a.split_k = p->split_k; a.k_chunk = p->k_chunk; a.partial = p->partial; a.ldp = p->ldp;
        a.batch = p->batch; a.stride_a = p->stride_a; a.stride_b = p->stride_b; a.stride_c = p->stride_c;
        if (ev) { cudaEventRecord(ev[0], s); cudaEventRecord(ev[1], s); }
        e = simt_launch(p->simt_id, a, s);
        if (ev) cudaEventRecord(ev[2], s);
        if (e == cudaSuccess && p->split_k > 1)
            e = splitk_reduce_launch(p->partial, p->split_k, p->M, p->N, p->ldp, C, p->ldc, s);
        if (ev) cudaEventRecord(ev[3], s);
        break;
    }
    case kCols: {
        ColsArgs a{};
        a.M = p->M; a.N = p->N; a.K = p->K;
        a.A = A; a.lda = p->lda; a.B = B; a.ldb = p->ldb; a.C = C; a.ldc = p->ldc;
        if (ev) { cudaEventRecord(ev[0], s); cudaEventRecord(ev[1], s); }
        e = cols_launch(a, p->num_sms, s);
        if (ev) { cudaEventRecord(ev[2], s); cudaEventRecord(ev[3], s); }
        break;
    }
    case kRows: {
        RowsArgs a{};
        a.M = p->M; a.N = p->N; a.K = p->K;
        a.A = A; a.lda = p->lda; a.B = B; a.ldb = p->ldb; a.C = C; a.ldc = p->ldc;
        a.partial = p->partial; a.ldp = p->ldp;
        a.range = p->k_chunk;
        if (ev) { cudaEventRecord(ev[0], s); cudaEventRecord(ev[1], s); }
        e = rows_launch(a, s);
        if (ev) cudaEventRecord(ev[2], s);
        if (e == cudaSuccess && p->split_k > 1)
            e = splitk_reduce_launch(p->partial, p->split_k, p->M, p->N, p->ldp, C, p->ldc, s);
        if (ev) cudaEventRecord(ev[3], s);
        break;
    }
    case kTc:
        e = tc_launch(p->tc, p->M, p->N, p->K, A, p->lda, B, p->ldb, C, p->ldc, p->d_status, s, ev);
        break;
    default:
        return GEMM_F32_ERR_INVALID_ARG;
    }
    return from_cuda(e);
}

gemm_f32_status gemm_f32_run_host(gemm_f32_plan_t p, const float* A_host, const float* B_host,
                                  float* C_host, gemm_f32_stream_t stream)
{
    if (!p) return GEMM_F32_ERR_INVALID_ARG;
    if (p->kind == kNoop) return GEMM_F32_OK;
    if (!C_host || (p->K > 0 && (!A_host || !B_host))) return GEMM_F32_ERR_INVALID_ARG;
    if (p->batch > 1) return GEMM_F32_ERR_UNSUPPORTED;
    if (!current_device_is(p->device)) return GEMM_F32_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t a_bytes = p->K > 0 ? size_t(p->M) * size_t(p->lda) * sizeof(float) : 0;
    const size_t b_bytes = p->K > 0 ? size_t(p->K) * size_t(p->ldb) * sizeof(float) : 0;
    const size_t c_bytes = size_t(p->M) * size_t(p->ldc) * sizeof(float);
    cudaError_t e = cudaSuccess;
    if (!p->hC) {
        if (a_bytes && (e = cudaMalloc(&p->hA, a_bytes)) != cudaSuccess) goto fail;
        if (b_bytes && (e = cudaMalloc(&p->hB, b_bytes)) != cudaSuccess) goto fail;
        if ((e = cudaMalloc(&p->hC, c_bytes)) != cudaSuccess) goto fail;
    }
    if (!p->xs[0]) {
        for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&p->xs[i], cudaStreamNonBlocking);
        for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&p->xev[i], cudaEventDisableTiming);
        if (e != cudaSuccess) return from_cuda(e);
    }
    if (const int panels = host_panel_count(p); panels > 1) {
        if ((e = make_panels(p, panels, host_col_width(p, panels))) != cudaSuccess ||
            (e = run_host_panels(p, A_host, B_host, C_host, s)) != cudaSuccess)
            return from_cuda(e);
        return gemm_f32_check(p, stream);
    }
    {
        // Each matrix is copied as two row halves on the two internal streams
        // (two copy engines at once); the caller's stream waits for both.
        auto fork = [&]() -> cudaError_t {
            cudaError_t r = cudaEventRecord(p->xev[0], s);
            for (int i = 0; i < 2 && r == cudaSuccess; ++i) r = cudaStreamWaitEvent(p->xs[i], p->xev[0], 0);
            return r;
        };
        auto join = [&]() -> cudaError_t {
            cudaError_t r = cudaSuccess;
            for (int i = 0; i < 2 && r == cudaSuccess; ++i) {
                r = cudaEventRecord(p->xev[1 + i], p->xs[i]);
                if (r == cudaSuccess) r = cudaStreamWaitEvent(s, p->xev[1 + i], 0);
            }
            return r;
        };
        auto halves = [&](float* dst, const float* src, int64_t rows, int64_t cols, int64_t ld,
                          cudaMemcpyKind kind) -> cudaError_t {
            const int64_t top = rows / 2;
            cudaError_t r = copy_rows(dst, src, top, cols, ld, kind, p->xs[0]);
            if (r == cudaSuccess)
                r = copy_rows(dst + top * ld, src + top * ld, rows - top, cols, ld, kind, p->xs[1]);
            return r;
        };
        if (p->K > 0) {
            if ((e = fork()) != cudaSuccess) return from_cuda(e);
            if ((e = halves(p->hA, A_host, p->M, p->K, p->lda, cudaMemcpyHostToDevice)) != cudaSuccess ||
                (e = halves(p->hB, B_host, p->K, p->N, p->ldb, cudaMemcpyHostToDevice)) != cudaSuccess ||
                (e = join()) != cudaSuccess)
                return from_cuda(e);
        }
        gemm_f32_status st = gemm_f32_run(p, p->hA, p->hB, p->hC, stream);
        if (st != GEMM_F32_OK) return st;
        if ((e = fork()) != cudaSuccess ||
            (e = halves(C_host, p->hC, p->M, p->N, p->ldc, cudaMemcpyDeviceToHost)) != cudaSuccess ||
            (e = join()) != cudaSuccess)
            return from_cuda(e);
    }
    return gemm_f32_check(p, stream);
fail:
    cudaGetLastError();
    cudaFree(p->hA); cudaFree(p->hB); cudaFree(p->hC);
    p->hA = p->hB = p->hC = nullptr;
    drop_panels(p);
    return from_cuda(e);
}

gemm_f32_status gemm_f32_check(gemm_f32_plan_t p, gemm_f32_stream_t stream)
{
    if (!p) return GEMM_F32_ERR_INVALID_ARG;
    if (p->kind == kNoop) return GEMM_F32_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return from_cuda(e);
    int h = 0;
    e = cudaMemcpy(&h, p->d_status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(e);
    if (h != kStatusOk) {
        e = cudaMemset(p->d_status, 0, sizeof(int));
        // a run that gave up may have left split-tile arrival counts behind
        if (e == cudaSuccess && p->kind == kTc && p->tc.sem_bytes) e = cudaMemset(p->tc.sem, 0, p->tc.sem_bytes);
        if (e == cudaSuccess && p->panel_sem) e = cudaMemset(p->panel_sem, 0, p->panel_sem_bytes);
        if (e != cudaSuccess) return from_cuda(e);
        return GEMM_F32_ERR_TIMEOUT;
    }
    return GEMM_F32_OK;
}

void gemm_f32_plan_destroy(gemm_f32_plan_t p)
{
    if (!p) return;
    for (cudaEvent_t e : p->trace_ev) cudaEventDestroy(e);
    if (p->ws) cudaFree(p->ws);
    if (p->hA) cudaFree(p->hA);
    if (p->hB) cudaFree(p->hB);
    if (p->hC) cudaFree(p->hC);
    for (cudaStream_t x : p->xs)
        if (x) cudaStreamDestroy(x);
    for (cudaEvent_t x : p->xev)
        if (x) cudaEventDestroy(x);
    drop_panels(p);
    for (cudaEvent_t x : p->pev) cudaEventDestroy(x);
    delete p;
}

gemm_f32_status gemm_f32_plan_describe(gemm_f32_plan_t p, char* buf, size_t n)
{
    if (!p || !buf || n == 0) return GEMM_F32_ERR_INVALID_ARG;
    snprintf(buf, n, "%s", p->desc);
    return GEMM_F32_OK;
}

size_t gemm_f32_plan_workspace_bytes(gemm_f32_plan_t p) { return p ? p->ws_bytes : 0; }

int gemm_f32_plan_kernel_launches(gemm_f32_plan_t p)
{
    if (!p) return -1;
    switch (p->kind) {
    case kZeroFill: return (int)p->batch;
    case kSimt: return p->split_k > 1 ? 2 : 1;
    case kRows: return p->split_k > 1 ? 2 : 1;
    case kCols: return 1;
    case kTc: {
        // the pre-pass (unless both operands are split in the kernel), the GEMM,
        // and the reduction of split tiles
        const int split = tc_config(p->tc.config_id).split;
        return (split == kSplitInKernel ? 1 : 2) + (p->tc.split_tiles > 0 && !p->tc.cluster && !p->tc.fixup ? 1 : 0);
    }
    default: return 0;
    }
}

gemm_f32_status gemm_f32_trace_enable(gemm_f32_plan_t p, int capacity)
{
    if (!p || capacity < 0) return GEMM_F32_ERR_INVALID_ARG;
    for (cudaEvent_t e : p->trace_ev) cudaEventDestroy(e);
    p->trace_ev.clear();
    p->trace_cap = p->trace_n = 0;
    if (capacity == 0 || p->kind == kNoop) return GEMM_F32_OK;
    try {
        p->trace_ev.resize(4 * size_t(capacity), nullptr);
    } catch (...) {
        return GEMM_F32_ERR_OOM;
    }
    for (cudaEvent_t& e : p->trace_ev) {
        cudaError_t r = cudaEventCreate(&e);
        if (r != cudaSuccess) {
            cudaGetLastError();
            for (cudaEvent_t x : p->trace_ev)
                if (x) cudaEventDestroy(x);
            p->trace_ev.clear();
            return from_cuda(r);
        }
    }
    p->trace_cap = capacity;
    return GEMM_F32_OK;
}

gemm_f32_status gemm_f32_trace_read(gemm_f32_plan_t p, float* ms, int max_runs, int* n_runs)
{
    if (!p || !n_runs || max_runs < 0 || (max_runs > 0 && !ms)) return GEMM_F32_ERR_INVALID_ARG;
    const int n = p->trace_n < max_runs ? p->trace_n : max_runs;
    for (int i = 0; i < n; ++i) {
        cudaEvent_t* ev = &p->trace_ev[4 * size_t(i)];
        cudaError_t r = cudaEventSynchronize(ev[3]);
        for (int j = 0; j < 3 && r == cudaSuccess; ++j) r = cudaEventElapsedTime(&ms[3 * i + j], ev[j], ev[j + 1]);
        if (r != cudaSuccess) return from_cuda(r);
    }
    *n_runs = n;
    p->trace_n = 0;
    return GEMM_F32_OK;
}

const char* gemm_f32_status_string(gemm_f32_status s)
{
    switch (s) {
    case GEMM_F32_OK: return "GEMM_F32_OK";
    case GEMM_F32_ERR_INVALID_ARG: return "GEMM_F32_ERR_INVALID_ARG";
    case GEMM_F32_ERR_UNSUPPORTED: return "GEMM_F32_ERR_UNSUPPORTED";
    case GEMM_F32_ERR_CUDA: return "GEMM_F32_ERR_CUDA";
    case GEMM_F32_ERR_TIMEOUT: return "GEMM_F32_ERR_TIMEOUT";
    case GEMM_F32_ERR_OOM: return "GEMM_F32_ERR_OOM";
    }
    return "GEMM_F32_ERR_UNKNOWN";
}

int gemm_f32_version(void) { return 200; }

}  // extern "C"
