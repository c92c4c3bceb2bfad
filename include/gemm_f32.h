/*
 * gemm_f32 — FP32 matrix multiply C = A*B on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the tiled dense FP32 GEMM whose K-loop stages tiles of A
 * and B through on-chip memory with a double-buffered / multi-stage prefetch
 * ("Double Buffering" technique page; "Case Study: The Double-Buffered GEMM",
 * its kernel listing and the paragraph on the single barrier's double duty).
 * Behind this interface:
 *
 *   - tcgen05 tensor-core kernels: a TMA producer warp fills an N-stage
 *     mbarrier ring in shared memory, an MMA warp accumulates into TMEM with an
 *     error-compensated 3xTF32 split, an epilogue warpgroup drains TMEM
 *     (TMA stores for each CTA's last tile); persistent over tiles, the last
 *     wave's tiles split into K-slices.  The operands are split into TF32
 *     pieces by a pre-pass kernel, or inside the GEMM kernel by converter
 *     warps, or half and half (see gemm_f32_opts.operand_split);
 *   - a SIMT FFMA kernel with cp.async double/multi-stage buffering (and an
 *     optional K split across the thread groups of a CTA), for small,
 *     latency-bound shapes and strided batches;
 *   - deterministic split-K reductions (a reduction kernel; optionally inside
 *     a thread-block cluster or by the last K-slice to arrive).
 *
 * A per-shape dispatcher chooses kernel, tile, stage count and split-K
 * ("Double Buffering" page, last paragraph, and the case study's first
 * paragraph: no single kernel is fastest; libraries dispatch per shape).
 *
 * Conventions (every entry point):
 *   - Row-major.  A is M x K with lda >= K, B is K x N with ldb >= N, C is
 *     M x N with ldc >= N; leading dimensions are in elements.
 *   - C is overwritten and never read (no alpha/beta): NaN in C before the
 *     call does not propagate.
 *   - M == 0 or N == 0: nothing to do, GEMM_F32_OK.  K == 0: C is filled with
 *     zeros (the empty sum).
 *   - A and B must not overlap C.  This is not checked.
 *   - Any base-pointer alignment and any leading dimension is accepted; the
 *     dispatcher routes around what a kernel cannot take.
 *   - Accuracy: for finite A and B with every S_ij = sum_k |A_ik||B_kj| below
 *     2^127, every element satisfies
 *         |C_ij - C_exact,ij| <= 2*K*2^-24*S_ij + K*2^-149 + t_ij.
 *     The first term is the usual bound of a K-term FP32 dot product.  The
 *     second is gradual underflow: each FP32 operation whose result falls
 *     below 2^-126 can be off by 2^-150, so it matters only for results or
 *     partial sums in the subnormal range.  t_ij = 0 for SIMT plans; for
 *     tensor-core plans t_ij = 2^-136 * sum_k (|B_kj| [0 < |A_ik| < 2^-113] +
 *     |A_ik| [0 < |B_kj| < 2^-113]): each operand is split into two TF32
 *     pieces, which resolve nothing finer than 2^-136 (TF32's smallest
 *     subnormal), so an element below 2^-113 is carried to within 2^-137.
 *     Subnormal operands are not flushed, and finite operands up to FLT_MAX
 *     stay finite through the split.  The two pieces carry 22 significand
 *     bits, whose per-product error of about 3*2^-22*|a||b| meets the first
 *     term only for K of about 10 and up, so the tensor-core path takes
 *     K >= 16 only; smaller K always runs on an FFMA kernel.  With
 *     non-finite inputs the affected outputs are non-finite, but not
 *     necessarily the IEEE value (the 3xTF32 split turns +-Inf into NaN).
 *   - Errors are returned as status codes; nothing calls exit or abort.
 *   - A plan is bound to the CUDA device that was current when it was made and
 *     must run with that device current.  One plan may be used from one stream
 *     at a time: it owns scratch memory (split-K partials, split operands).
 *     Different plans may run on different streams at once.
 *   - gemm_f32_run only enqueues kernels on the stream and allocates nothing,
 *     so its runs can be captured in a CUDA graph (after one plain run of the
 *     plan, which sets the kernels' attributes); gemm_f32_run_host and
 *     gemm_f32_check synchronise and cannot.
 */
#ifndef GEMM_F32_H_
#define GEMM_F32_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_F32_API __attribute__((visibility("default")))
#else
#define GEMM_F32_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque plan.  Created by gemm_f32_plan / gemm_f32_plan_ex, owned by the
 * caller, released by gemm_f32_plan_destroy. */
typedef struct gemm_f32_plan_s* gemm_f32_plan_t;

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* gemm_f32_stream_t;

typedef enum {
    GEMM_F32_OK = 0,
    GEMM_F32_ERR_INVALID_ARG = 1, /* bad size, leading dimension, NULL pointer or option */
    GEMM_F32_ERR_UNSUPPORTED = 2, /* forced variant cannot run this problem; no GPU of the right kind */
    GEMM_F32_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, copy, tensor map) */
    GEMM_F32_ERR_TIMEOUT = 4,     /* a kernel's bounded wait ran out; the result is not valid */
    GEMM_F32_ERR_OOM = 5          /* device or pinned host allocation failed */
} gemm_f32_status;

typedef enum {
    GEMM_F32_VARIANT_AUTO = 0,     /* dispatcher's choice */
    GEMM_F32_VARIANT_SIMT = 1,     /* FFMA, cp.async multi-stage */
    GEMM_F32_VARIANT_TCGEN05 = 2,  /* tcgen05 3xTF32 with TMA/mbarrier pipeline */
    GEMM_F32_VARIANT_SHORT_M = 3,  /* FFMA for M <= 16 (else UNSUPPORTED): B streamed once in
                                      256-column blocks over ranges of K, the ranges' sums
                                      added by the split-K reduction; the dispatcher takes it
                                      for M <= 8 with K x N at least 2^24 */
    GEMM_F32_VARIANT_SHORT_N = 4   /* FFMA for N <= 16 (else UNSUPPORTED): a warp per row of C
                                      streams that row of A once, its lanes' sums added in a
                                      fixed order; fast for N = 1 only, where the dispatcher
                                      takes it (M at least 4096, M x K at least 2^24) */
} gemm_f32_variant;

/* Options for gemm_f32_plan_ex.  Zero means "dispatcher's choice" for every
 * field; gemm_f32_opts_init fills the defaults. */
typedef struct {
    int32_t variant;        /* gemm_f32_variant */
    int32_t tile_m;         /* output tile rows (SIMT: 32/64/128; TC: 128, or 256 = one tile per pair
                               of CTAs, a thread-block cluster of two sharing each tcgen05.mma
                               (cta_group::2): operand_split 2 to 5 (not the full pre-pass),
                               tile_n 128 or 256, tile_k 32 or 16 (16: in the kernel, or with
                               operand_split 4 at tile_n 256); needs K >= 32 and lda a multiple
                               of 4 (ldb too when B is split in the kernel), else UNSUPPORTED;
                               a base pointer the TMA cannot take runs the one-CTA pre-pass form
                               instead) */
    int32_t tile_n;         /* output tile cols (SIMT: 32/64/128; TC: 64/128/256) */
    int32_t stages;         /* pipeline depth (SIMT: 1..4; TC: 2..8) */
    int32_t split_k;        /* K splits, 1 = none (max 64) */
    int32_t tf32_terms;     /* TC only: 3 = 3xTF32 (default); 1 = single TF32 product,
                               a deliberately inaccurate negative control for tests */
    int64_t wait_timeout_cycles; /* TC only: limit of every device-side wait, in SM clock
                                    cycles; 0 = default (about 2^32 cycles) */
    int32_t debug_withhold_stage; /* TC only, test hook: >0 makes the producer skip the
                                     load of that pipeline fill (1-based), so the MMA
                                     warp's bounded wait runs out and the run reports
                                     GEMM_F32_ERR_TIMEOUT through gemm_f32_check */
    int32_t separate_syncs; /* ablation of the pages' barrier coalescing: 1 publishes A and
                               B through separate synchronisations (SIMT: one barrier after
                               each operand's copy; TC: separate "full" mbarriers for A and
                               B); 0 = one synchronisation for both (default) */
    int32_t operand_split;  /* TC only: where the 3xTF32 split happens.  0 = dispatcher's
                               choice; 1 = a pre-pass writes hi/lo operands to scratch;
                               2 = inside the GEMM kernel (needs K >= 32 and lda, ldb
                               multiples of 4); 3 = A inside the kernel, B by the pre-pass
                               (needs K >= 32, lda a multiple of 4); 4 = hi of A read from
                               A itself, lo of A and B by the pre-pass (same needs; on CTA
                               pairs this form has no conversion inside the kernel); 5 = CTA
                               pairs only (tile 256x256, tile_k 32): raw A staged by TMA in a
                               short ring, split by the kernel's loader warps into tensor
                               memory, B by the pre-pass (same needs; measured slower than
                               4, never the dispatcher's choice).  2 to 5
                               fall back to 1 at run time for a base pointer of A (or, for 2,
                               B) that is not 16-byte aligned */
    int32_t tile_group;     /* TC only: tile order of the persistent kernel, in tile-rows per
                               raster group (1..64; 0 = the dispatcher's choice, else 8) */
    int32_t tile_k;         /* K-tile depth.  SIMT: 16/32/64 (0 = the compiled default for the
                               tile and stage count).  tcgen05: 32, or 16 for half-size,
                               twice-as-deep stages of the in-kernel split (selects that
                               form) or of the CTA-pair form with operand_split 4; 0 = the
                               dispatcher's choice */
    int32_t host_panels;    /* TC only, gemm_f32_run_host: row panels the host-buffer run is
                               pipelined over (A panel copies, panel GEMMs and C panel
                               copies overlap); 0 = the dispatcher's choice, 1 = none,
                               n = n panels of whole tiles (128 rows; 256 for CTA-pair plans;
                               at most 64); with column blocks on a GEMM of 8 waves or more
                               the first panel takes two shares of the tile rows; with column
                               blocks and three panels or more, the last panel runs as two
                               column halves when each half holds a wave of tiles, the first
                               half's C copied back while the second half's GEMM runs */
    int32_t split_reduce;   /* TC only: how the K-slices of split tiles are summed.  0 = the
                               dispatcher's choice (1: measured fastest); 1 = a
                               reduction kernel over partial tiles in scratch; 3 = no extra
                               launch: every slice stores its partial tile, and the last slice
                               of each tile to arrive (an atomic count per 32-row quadrant) sums
                               them in slice order and writes C (needs at most 8 slices, at most
                               one wave of split units and a ring of 144 KB or more; else
                               UNSUPPORTED); 2 = the
                               slices of a tile run as one cluster of 2 or 4 CTAs and sum in
                               distributed shared memory (needs every tile split in 2 or 4,
                               all slices resident at once, tiles at most 128 wide and a ring
                               of 128 KB or more; else UNSUPPORTED); 4 = CTA pairs (tile_m 256,
                               operand_split 2 to 4) only: the kernel's grid, launched
                               cooperatively, passes a grid-wide barrier once every unit is
                               stored and then sums the slices itself, in the reduction
                               kernel's order (bit-identical; no reduction launch) */
    int32_t k_slices;       /* SIMT only: thread groups of a CTA that split each K-tile between
                               them and add their register tiles at the end (1, 2 or 4; 0 = the
                               dispatcher's choice): more warps per SM for small grids without a
                               second launch */
    int32_t host_col_blocks; /* TC only, gemm_f32_run_host with two or more row panels: the
                               first row panel runs as this many column blocks of whole tiles,
                               B copied block by block, each block's GEMM starting as soon as
                               its columns of B have landed (the GEMM starts after a fraction
                               of B instead of all of it).  0 = the dispatcher's choice, 1 =
                               none, at most 16; only for plans that split A inside the GEMM
                               kernel or read hi of A from A (operand_split 2 to 5),
                               otherwise as 1 */
    int32_t simt_fragments;  /* SIMT only: how each thread's register fragments come from the
                               staged tiles.  0 = 16-byte shared-memory loads that lanes
                               needing the same values share (broadcast; default); 1 = each
                               distinct value read once per warp and handed to the lanes by
                               warp shuffles (an ablation, compiled for a few tiles only;
                               UNSUPPORTED elsewhere) */
} gemm_f32_opts;

/* Fill *opts with the defaults (all zero). INVALID_ARG if opts is NULL. */
GEMM_F32_API gemm_f32_status gemm_f32_opts_init(gemm_f32_opts* opts);

/*
 * Make a plan for C[M x N] = A[M x K] * B[K x N] with the given leading
 * dimensions: the product the pages' tiled kernel computes ("Case Study: The
 * Double-Buffered GEMM", its kernel listing: each output tile is the sum, over
 * the K-tiles staged in on-chip memory, of the products of A's row panel and
 * B's column panel).  The plan fixes what that kernel takes besides the
 * matrices: the sizes, and here the leading dimensions.  Chooses the kernel and its configuration, allocates the plan's
 * scratch memory on the current device (cudaMalloc) and prepares the tensor
 * maps of that scratch.  Pointers to A, B and C are given only at run time.
 *
 * INVALID_ARG: M, N or K negative; lda < K, ldb < N or ldc < N (when the
 * matrix is non-empty); leading dimension < 1; plan NULL.
 * UNSUPPORTED: no CUDA device, or the device is not sm_103.
 * OOM: scratch allocation failed.  On any error *plan is set to NULL.
 */
GEMM_F32_API gemm_f32_status gemm_f32_plan(int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldc,
                              gemm_f32_plan_t* plan);

/* As gemm_f32_plan, with options (NULL = defaults).  A forced variant or
 * configuration that cannot run the problem gives UNSUPPORTED or INVALID_ARG. */
GEMM_F32_API gemm_f32_status gemm_f32_plan_ex(int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int64_t ldc,
                                 const gemm_f32_opts* opts, gemm_f32_plan_t* plan);

/*
 * Plan `batch` independent products of the same shape, run by one launch:
 * C_z = A_z * B_z for z = 0 .. batch-1, with A_z = A + z*stride_a,
 * B_z = B + z*stride_b, C_z = C + z*stride_c (strides in elements; 0 for A or
 * B reuses one operand for every product).  Many small GEMMs in one launch pay
 * the launch latency once; the pages tie such small, latency-dominated
 * products to the decode regime ("Case Study: The Double-Buffered GEMM", the
 * three-regimes paragraph).  Runs on the SIMT kernel (no split-K).  gemm_f32_run
 * takes the base pointers A, B, C of product 0.
 *
 * INVALID_ARG: as gemm_f32_plan; batch < 0 or > 65535; a negative stride; or
 * stride_c smaller than one C (the outputs would overlap).  batch == 0 is an
 * empty problem.  opts may be NULL; its variant must be AUTO or SIMT.
 */
GEMM_F32_API gemm_f32_status gemm_f32_plan_batched(int64_t M, int64_t N, int64_t K,
                                                   int64_t lda, int64_t ldb, int64_t ldc,
                                                   int64_t batch, int64_t stride_a, int64_t stride_b,
                                                   int64_t stride_c, const gemm_f32_opts* opts,
                                                   gemm_f32_plan_t* plan);

/*
 * Enqueue C = A*B on `stream`: one pass of the pipelined K-loop over every
 * output tile ("Double Buffering" technique page: the next K-tile is fetched
 * while the current one is multiplied, one synchronisation per K-tile
 * publishing the copy and freeing the buffer it will overwrite; "Case Study:
 * The Double-Buffered GEMM", kernel listing).  A, B, C are device pointers
 * with the plan's shapes and leading dimensions.  Asynchronous: returns after the launches are
 * queued; nothing is synchronised.  INVALID_ARG for a NULL plan or a NULL
 * pointer with non-empty work; CUDA if a launch fails.  A device-side timeout
 * is reported later by gemm_f32_check.
 */
GEMM_F32_API gemm_f32_status gemm_f32_run(gemm_f32_plan_t plan, const float* A, const float* B,
                             float* C, gemm_f32_stream_t stream);

/*
 * C = A*B with HOST operands: copies A and B to device buffers the plan owns
 * (allocated on first use), runs, copies C back to host memory and
 * synchronises `stream`.  For pinned host memory the copies are asynchronous
 * DMA; pageable memory works but is slower.  Tensor-core plans with enough
 * tiles run as a pipeline over row panels of A and C: B is copied and split
 * once, then each panel's GEMM overlaps the next panel's A copy and the
 * previous panel's C copy (two internal streams, ordered by events after
 * `stream`'s earlier work).  Returns the run's status, or TIMEOUT if a
 * device-side wait ran out; UNSUPPORTED for a batched plan.
 */
GEMM_F32_API gemm_f32_status gemm_f32_run_host(gemm_f32_plan_t plan, const float* A_host,
                                  const float* B_host, float* C_host,
                                  gemm_f32_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the plan's device status word.
 * TIMEOUT if a kernel of an earlier run gave up a bounded wait (that run's C
 * is not valid); CUDA if the stream reports an error; OK otherwise.
 */
GEMM_F32_API gemm_f32_status gemm_f32_check(gemm_f32_plan_t plan, gemm_f32_stream_t stream);

/* Release the plan and its scratch memory.  NULL is a no-op.  The caller must
 * make sure no run of this plan is still executing. */
GEMM_F32_API void gemm_f32_plan_destroy(gemm_f32_plan_t plan);

/* Write a one-line, NUL-terminated description of the chosen configuration
 * (variant, tile, stages, split-K, scratch bytes) into buf[0..n-1].
 * INVALID_ARG for a NULL plan or buffer or n == 0. */
GEMM_F32_API gemm_f32_status gemm_f32_plan_describe(gemm_f32_plan_t plan, char* buf, size_t n);

/* Bytes of device scratch the plan holds (0 for none). */
GEMM_F32_API size_t gemm_f32_plan_workspace_bytes(gemm_f32_plan_t plan);

/* Number of kernels one gemm_f32_run of this plan launches (0 for an empty
 * problem), or -1 for a NULL plan. */
GEMM_F32_API int gemm_f32_plan_kernel_launches(gemm_f32_plan_t plan);

/*
 * Kernel-level timing with CUDA events (tracing).  After
 * gemm_f32_trace_enable(plan, capacity) each of the next `capacity` runs
 * records four events on its stream, at the boundaries of its three phases:
 * operand split (tensor-core path only), main GEMM kernel, split-K reduction.
 * gemm_f32_trace_read waits for the recorded events, writes the phase
 * durations in milliseconds to ms[3*i + 0..2] for run i (0 for a phase the
 * run does not have), sets *n_runs, and empties the record.  capacity 0
 * disables tracing.  The plan creates the events (cudaEventCreate) when
 * tracing is enabled.  INVALID_ARG for a NULL plan, a negative capacity or
 * NULL outputs; CUDA if an event call fails.
 */
GEMM_F32_API gemm_f32_status gemm_f32_trace_enable(gemm_f32_plan_t plan, int capacity);
GEMM_F32_API gemm_f32_status gemm_f32_trace_read(gemm_f32_plan_t plan, float* ms, int max_runs,
                                                 int* n_runs);

/*
 * C = A*B without allocating anything.  (An addition of this library; the
 * pages have no counterpart.)
 *
 * For callers that cannot allocate device memory when they need the product:
 * code running while an allocator or memory pool is being set up or torn down,
 * code whose device memory all comes from an arena it manages itself, or a
 * latency-critical path that must not take the allocator's locks.
 * gemm_f32_plan allocates its scratch with cudaMalloc; this call does not.
 *
 * It runs the SIMT FFMA kernel with K split into `split_k` slices (2..64),
 * followed by the deterministic split-K reduction.  The slices hold whole
 * 16-deep K-tiles, so s = ceil(K / (16 * ceil(ceil(K / split_k) / 16))) of
 * them run (s <= split_k; s = 1 for K <= 16, which writes C directly and
 * uses no scratch).  The partial products of s > 1 slices live in one fixed
 * 8 MiB array inside the library image, which every GPU that loads the
 * library holds until the process exits; the call needs s * M * round_up(N, 4)
 * floats of it and returns INVALID_ARG when that exceeds 2^21 floats (8 MiB).
 * Nothing in the call runs cudaMalloc, cudaFree or any other allocating
 * routine.
 *
 * A, B, C are device pointers with the layout of the conventions above; the
 * call is asynchronous on `stream`.  Each call that uses the array looks up
 * its device address in the current context (cudaGetSymbolAddress, which
 * allocates nothing), so the address stays right even if the device's
 * context is destroyed and created again.  The first such call on a device
 * also makes the library's device code resident there: make it before any
 * stream capture.  All calls share the one array and each overwrites what
 * the last one left; every partial is written in full before it is read, so
 * nothing has to start at zero.  Calls whose executions overlap on the GPU
 * (different streams, or several host threads) race on the array and give
 * wrong results: serialise them.
 *
 * INVALID_ARG: bad sizes or leading dimensions, split_k outside 2..64, NULL
 * pointers with non-empty work, or partials larger than the array.
 * UNSUPPORTED: the current device is not sm_103.  CUDA: a launch failed.
 * M == 0 or N == 0 returns OK at once; K == 0 writes zeros to C.
 */
GEMM_F32_API gemm_f32_status gemm_f32_run_splitk_noalloc(int64_t M, int64_t N, int64_t K,
                                                         int64_t lda, int64_t ldb, int64_t ldc,
                                                         const float* A, const float* B, float* C,
                                                         int32_t split_k, gemm_f32_stream_t stream);

/* Static, NUL-terminated name of a status code. */
GEMM_F32_API const char* gemm_f32_status_string(gemm_f32_status s);

/* Library version: major*10000 + minor*100 + patch. */
GEMM_F32_API int gemm_f32_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F32_H_ */
