// tcgen05 3xTF32 GEMM that splits the operands inside the kernel.
//
// Same pipeline as tc_gemm.cu ("Double Buffering" technique page and "Case
// Study: The Double-Buffered GEMM": the next tile is fetched while the current
// one is multiplied), but the TMA engine copies the caller's raw FP32 A and B
// tiles, so no split pre-pass and no split operands in HBM are needed:
//
//   * A arrives K-major in the 128-byte swizzled layout the MMA reads.  A
//     kind::tf32 MMA uses the top 19 bits of each FP32 operand (measured on
//     GB300: it truncates), so the raw tile itself is hi_A = trunc_tf32(A).
//     Converter warps add lo_A = A - hi_A rounded to TF32 beside it, element by
//     element in the same swizzled layout.
//   * B arrives N-major (B is row-major K x N) as 32 x 32 boxes.  Converter
//     warps transpose it to the K-major swizzled layout as hi_B (the raw value,
//     truncated by the MMA) and lo_B = B - trunc_tf32(B) rounded to TF32.
//
// With this truncation split each product carries up to about 2^-19*|a||b|
// of error (hi_A*lo_B + lo_A*hi_B + hi_A*hi_B drops lo_A*lo_B < 2^-20|ab| and
// rounds each lo to 11 bits), which meets the FP32 bound 2*K*2^-24*sum|a||b|
// for K >= 32; plans take this kernel only then.
//
// A hybrid form takes B already split and transposed by the pre-pass (hi/lo
// copied straight into the slot) and converts only A in the kernel: half the
// pre-pass, and a quarter of the converters' shared-memory traffic.
//
// Shared memory: SLOTS MMA-facing slots [A_raw | lo_A | hi_B | lo_B].  Raw B
// (32 x 32 boxes, N-major) lands in the lo_B part of its own slot: the
// converters read it into registers, write hi_B beside it, agree that every
// warp has read (the slot's `rd` barrier), then write lo_B over it.  So B's
// copy recycles with the slot, as deep as the ring, instead of through
// separate staging buffers.  Barriers per slot: full (A and raw B landed), rd
// (every converter warp holds its raw B), conv (converters done: hi/lo of A
// and B ready), empty (MMAs done).
//
// Roles (448 threads, one CTA per SM, persistent over units of work):
//   warp 0      TMA producer           warp 1      TMEM allocator + MMA issuer
//   warps 2..5  epilogue (TMEM lanes 32*(w%4)..)   warps 6..13 converters
// Every wait is bounded as in tc_gemm.cu (timeout -> status word, abort flag,
// drain, TMEM freed).
#include <cstdint>

#include "tc_common.cuh"

namespace gemm_f32 {
namespace {

using namespace tc;
constexpr int kConvWarps = 8;                       // one per 4-wide k group of a 32-k block
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kFusedThreads = 6 * 32 + kConvThreads;

// KB: k per pipeline stage.  32 = one 128-byte swizzled row of FP32 per operand
// row (the same layout as the pre-split operands); 16 = half-size stages in
// the 64-byte swizzled layout, twice as many of them in the same shared memory.
template <int BN, int SLOTS, bool BPRE, int KB>
struct FusedLayout {
    static constexpr int A_BYTES = kBM * KB * 4;           // 16 KB (KB 32), 8 KB (KB 16)
    static constexpr int B_BYTES = BN * KB * 4;            // also raw B: BN/32 boxes of KB k x 32 n
    static constexpr int BOX_BYTES = 32 * KB * 4;          // one raw-B box
    static_assert(KB == 32 || KB == 16, "stage depth");
    static_assert(B_BYTES == BN / 32 * BOX_BYTES, "raw B fills the lo_B part exactly");
    static_assert(!BPRE || KB == 32, "pre-split B comes in 32-k rows");
    static constexpr int SLOT_BYTES = 2 * A_BYTES + 2 * B_BYTES;
    static constexpr int RING_BYTES = SLOTS * SLOT_BYTES;
    // full, rd, conv, empty per slot + tmem full/empty x2, drain, ready, recv,
    // stg, sumd, fixup loads x4
    static constexpr int NBARS = 4 * SLOTS + 13;
    static constexpr bool FIXUP_OK = kFixRingBytes <= RING_BYTES;
    // cluster K-slice sum: its staging and receive buffers laid over the idle ring
    static constexpr bool CLUSTER_OK = ClusterSum<BN>::BYTES <= RING_BYTES;
    static constexpr int BAR_BYTES = 8 * NBARS + 16;
    static constexpr int SMEM_USED = 1024 + RING_BYTES + BAR_BYTES;
    static constexpr int SMEM_BYTES = SMEM_USED > 116 * 1024 ? SMEM_USED : 116 * 1024;
    static constexpr uint32_t TMEM_COLS = 2 * BN;
    static_assert(BN % 32 == 0 && BN <= 256, "B arrives in 32-column boxes");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

template <int BN, int SLOTS, bool BPRE, int KB>
constexpr bool L_STAGING_FITS = FusedLayout<BN, SLOTS, BPRE, KB>::RING_BYTES >= 4 * 8192;

// Byte offset of the 16-byte chunk kq of row `row` in a K-major swizzled tile:
// KB 32: rows of 128 B in 8-row atoms of 1024 B, chunk index XOR row % 8;
// KB 16: rows of 64 B in 8-row atoms of 512 B, chunk index XOR (row / 2) % 4
// (the 64-byte swizzle: byte-address bits 4-5 XOR bits 7-8).
template <int KB>
__device__ __forceinline__ uint32_t kmajor_off(int row, int kq)
{
    if constexpr (KB == 32)
        return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((kq ^ (row & 7)) << 4));
    else
        return (uint32_t)((row >> 3) * 512 + (row & 7) * 64 + ((kq ^ ((row >> 1) & 3)) << 4));
}

// Shared-memory matrix descriptor of a K-major operand in the layout above.
template <int KB>
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr)
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

// BPRE is the hybrid form: B comes already split (hi/lo, K-major) from the
// pre-pass through tm_bhi/tm_blo, straight into the slot, and the converters
// only add lo_A.  Otherwise tm_b copies raw B into the slot's lo_B part.
template <int BN, int SLOTS, bool BPRE, int KB>
__global__ void __launch_bounds__(kFusedThreads, 1)
tc_fused_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_bhi, const __grid_constant__ CUtensorMap tm_blo,
                const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_p,
                const TcArgs args)
{
    using L = FusedLayout<BN, SLOTS, BPRE, KB>;
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
    auto full_a = [&](int s) { return ptx::smem_u32(bars + s); };
    auto conv = [&](int s) { return ptx::smem_u32(bars + SLOTS + s); };
    auto empty = [&](int s) { return ptx::smem_u32(bars + 2 * SLOTS + s); };
    auto rd = [&](int s) { return ptx::smem_u32(bars + 3 * SLOTS + s); };
    auto tfull = [&](int b) { return ptx::smem_u32(bars + 4 * SLOTS + b); };
    auto tempty = [&](int b) { return ptx::smem_u32(bars + 4 * SLOTS + 2 + b); };
    const uint32_t drain_bar = ptx::smem_u32(bars + 4 * SLOTS + 4);
    const uint32_t ready_bar = ptx::smem_u32(bars + 4 * SLOTS + 5);
    const uint32_t recv_bar = ptx::smem_u32(bars + 4 * SLOTS + 6);
    const uint32_t stg_bar = ptx::smem_u32(bars + 4 * SLOTS + 7);
    const uint32_t sum_bar = ptx::smem_u32(bars + 4 * SLOTS + 8);
    auto fix_bar = [&](int q) { return ptx::smem_u32(bars + 4 * SLOTS + 9 + q); };
    const bool clustered = L::CLUSTER_OK && args.cluster > 1;
    const bool fixup = L::FIXUP_OK && args.fixup && !clustered;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SLOTS; ++s) {
            ptx::mbar_init(full_a(s), 1);
            ptx::mbar_init(conv(s), kConvThreads / 32);
            ptx::mbar_init(empty(s), 1);
            ptx::mbar_init(rd(s), kConvThreads / 32);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull(b), 1);
            ptx::mbar_init(tempty(b), 4);
        }
        ptx::mbar_init(drain_bar, 1);
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
        ptx::tma_prefetch_desc(&tm_a);
        if (BPRE) {
            ptx::tma_prefetch_desc(&tm_bhi);
            ptx::tma_prefetch_desc(&tm_blo);
        } else {
            ptx::tma_prefetch_desc(&tm_b);
        }
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
    // Programmatic launch: only the producer reads global memory first, so only
    // it waits for the previous kernel on the stream (below); the next kernel
    // may start its own prologue now.
    pdl_trigger();

    const int num_work = args.dp_tiles + args.split_tiles * args.splits;
    const int64_t limit = args.timeout;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            pdl_wait();  // the previous kernel's writes (A, B, C) are done
            uint32_t fills = 0;
            bool stop = false;
            for (int w = blockIdx.x; w < num_work && !stop; w += gridDim.x) {
                const Unit u = decode_unit(w, args);
                int tm, tn;
                tile_coords(u.tile, args.tiles_m, args.tiles_n, args.group, tm, tn);
                for (int kh = u.kb0 * HALVES; kh < u.kb1 * HALVES; ++kh) {
                    const int s = fills % SLOTS;
                    const uint32_t ps = (fills / SLOTS) & 1u;
                    if (!wait_phase(empty(s), ps ^ 1u, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
                    const int kc = kh * KB;
                    const uint32_t slot = ring + s * L::SLOT_BYTES;
                    if constexpr (BPRE) {
                        ++fills;
                        if (fills == (uint32_t)args.withhold) continue;
                        ptx::mbar_arrive_expect_tx(full_a(s), L::A_BYTES + 2 * L::B_BYTES);
                        ptx::tma_load_2d(slot, &tm_a, full_a(s), kc, tm * kBM);
                        ptx::tma_load_2d(slot + 2 * L::A_BYTES, &tm_bhi, full_a(s), kc, tn * BN);
                        ptx::tma_load_2d(slot + 2 * L::A_BYTES + L::B_BYTES, &tm_blo, full_a(s), kc, tn * BN);
                    } else {
                        ++fills;
                        if (fills == (uint32_t)args.withhold) continue;
                        // raw A into the A part, raw B boxes into the lo_B part
                        ptx::mbar_arrive_expect_tx(full_a(s), L::A_BYTES + L::B_BYTES);
                        ptx::tma_load_2d(slot, &tm_a, full_a(s), kc, tm * kBM);
#pragma unroll
                        for (int j = 0; j < BN / 32; ++j)
                            ptx::tma_load_2d(slot + 2 * L::A_BYTES + L::B_BYTES + j * L::BOX_BYTES, &tm_b,
                                             full_a(s), tn * BN + 32 * j, kc);
                    }
                }
            }
            // Drain: the last fill of every slot must have landed.
            const uint32_t total = fills;
            auto drain = [&](uint32_t bar_of_last, uint32_t last, int depth) {
                if (last + 1 == (uint32_t)args.withhold) return;
                const uint32_t par = (last / depth) & 1u;
                const long long t0 = clock64();
                while (!ptx::mbar_try_wait(bar_of_last, par))
                    if (clock64() - t0 > limit) { atomicExch(args.status, kStatusTimeout); break; }
            };
            for (int s = 0; s < SLOTS && (uint32_t)s < total; ++s)
                drain(full_a(s), (total - 1 - s) / SLOTS * SLOTS + s, SLOTS);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_tf32<BN>();
            uint32_t fills = 0;
            int iter = 0;
            bool stop = false;
            for (int w = blockIdx.x; w < num_work && !stop; w += gridDim.x, ++iter) {
                const Unit u = decode_unit(w, args);
                const int buf = iter & 1;
                const uint32_t tphase = (iter >> 1) & 1;
                if (!wait_phase(tempty(buf), tphase ^ 1u, limit, abort_flag, args.status)) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kh = u.kb0 * HALVES; kh < u.kb1 * HALVES; ++kh, ++fills) {
                    const int s = fills % SLOTS;
                    const uint32_t ps = (fills / SLOTS) & 1u;
                    if (!wait_phase(conv(s), ps, limit, abort_flag, args.status)) {
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
                            ptx::mma_tf32(d_tmem, kmajor_desc<KB>(a_lo + off), kmajor_desc<KB>(b_hi + off), idesc, acc);
                            ptx::mma_tf32(d_tmem, kmajor_desc<KB>(a_hi + off), kmajor_desc<KB>(b_lo + off), idesc, 1u);
                            ptx::mma_tf32(d_tmem, kmajor_desc<KB>(a_hi + off), kmajor_desc<KB>(b_hi + off), idesc, 1u);
                        } else {
                            ptx::mma_tf32(d_tmem, kmajor_desc<KB>(a_hi + off), kmajor_desc<KB>(b_hi + off), idesc, acc);
                        }
                    }
                    ptx::mma_commit(empty(s));
                }
                if (stop) break;
                ptx::mma_commit(tfull(buf));
            }
            ptx::mma_commit(drain_bar);
            const long long t0 = clock64();
            while (!ptx::mbar_try_wait(drain_bar, 0))
                if (clock64() - t0 > limit) { atomicExch(args.status, kStatusTimeout); break; }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------ epilogue ------------------------------
        const int quad = warp & 3;
        int iter = 0;
        for (int w = blockIdx.x; w < num_work; w += gridDim.x, ++iter) {
            const Unit u = decode_unit(w, args);
            int tm, tn;
            tile_coords(u.tile, args.tiles_m, args.tiles_n, args.group, tm, tn);
            const int buf = iter & 1;
            const uint32_t tphase = (iter >> 1) & 1;
            if (!wait_phase(tfull(buf), tphase, limit, abort_flag, args.status)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + buf * BN;
            const EpilogueBars eb{ready_bar, recv_bar, stg_bar, sum_bar, fix_bar(quad)};
            if (!drain_unit<BN, L::RING_BYTES>(args, &tm_c, &tm_p, u, tm, tn, taddr, quad, lane,
                                               w + (int)gridDim.x >= num_work, clustered, fixup, ring, ring_ptr, eb,
                                               limit, abort_flag))
                break;
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty(buf));
        }
    } else {
        // ------------------------------ converters ----------------------------
        const int ct = threadIdx.x - 6 * 32;  // 0 .. kConvThreads-1
        constexpr int KG = KB / 4;            // 4-wide k groups per stage
        constexpr int PARTS = kConvWarps / KG;  // warps per k group: they share the boxes
        const int cw = (ct >> 5) % KG;        // k group of this warp: k = 4*cw .. 4*cw+3
        const int part = (ct >> 5) / KG;      // boxes part, part + PARTS, ...
        uint32_t fills = 0;
        bool stop = false;
        // Offsets inside a raw-B box (rows of 32 n, 128-byte swizzled) of the four
        // k rows this lane reads (row k, chunk (lane/4) ^ (k%8), word lane%4).
        uint32_t box_off[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = cw * 4 + j;
            box_off[j] = (uint32_t)(k * 128 + (((lane >> 2) ^ (k & 7)) << 4) + (lane & 3) * 4);
        }
        for (int w = blockIdx.x; w < num_work && !stop; w += gridDim.x) {
            const Unit u = decode_unit(w, args);
            for (int kh = u.kb0 * HALVES; kh < u.kb1 * HALVES; ++kh, ++fills) {
                const int s = fills % SLOTS;
                const uint32_t ps = (fills / SLOTS) & 1u;
                if (!wait_phase(full_a(s), ps, limit, abort_flag, args.status)) {
                    stop = true;
                    break;
                }
                uint8_t* slot = ring_ptr + s * L::SLOT_BYTES;
                const uint8_t* a_raw = slot;
                uint8_t* a_lo = slot + L::A_BYTES;
                uint8_t* b_hi = slot + 2 * L::A_BYTES;
                uint8_t* b_lo = b_hi + L::B_BYTES;  // holds raw B until every warp has read it
                // B: this warp's raw values (k = 4*cw..4*cw+3, n = lane of its
                // 32-column boxes) into registers; hi_B written at once.  The
                // reads of a box row are conflict-free, and the 16-byte writes of
                // 8 consecutive rows land in 8 different swizzled chunks.
                constexpr int NBW = BPRE ? 1 : BN / 32 / PARTS;  // boxes per warp
                float v[NBW][4];
                if constexpr (!BPRE) {
#pragma unroll
                    for (int i = 0; i < NBW; ++i) {
                        const int nb = part + i * PARTS;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            v[i][j] = *reinterpret_cast<const float*>(b_lo + nb * L::BOX_BYTES + box_off[j]);
                        *reinterpret_cast<float4*>(b_hi + kmajor_off<KB>(nb * 32 + lane, cw)) =
                            make_float4(v[i][0], v[i][1], v[i][2], v[i][3]);
                    }
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(rd(s));
                }
                // A: lo beside the raw tile, same swizzled position, 16 bytes at a time.
#pragma unroll
                for (int c = ct; c < L::A_BYTES / 16; c += kConvThreads) {
                    const float4 x = *reinterpret_cast<const float4*>(a_raw + c * 16);
                    *reinterpret_cast<float4*>(a_lo + c * 16) =
                        make_float4(lo_part(x.x), lo_part(x.y), lo_part(x.z), lo_part(x.w));
                }
                if constexpr (!BPRE) {
                    // every warp holds its raw B: lo_B may overwrite it
                    if (!wait_phase(rd(s), ps, limit, abort_flag, args.status)) {
                        stop = true;
                        break;
                    }
#pragma unroll
                    for (int i = 0; i < NBW; ++i)
                        *reinterpret_cast<float4*>(b_lo + kmajor_off<KB>((part + i * PARTS) * 32 + lane, cw)) =
                            make_float4(lo_part(v[i][0]), lo_part(v[i][1]), lo_part(v[i][2]), lo_part(v[i][3]));
                }
                ptx::fence_proxy_async_shared();  // generic-proxy writes -> tensor core reads
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(conv(s));
            }
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

template <int BN, int SLOTS, bool BPRE, int KB>
cudaError_t launch_fused(const TcPlanState& st, const TcArgs& a, const CUtensorMap& ta, const CUtensorMap& tb,
                         const CUtensorMap& tbhi, const CUtensorMap& tblo, cudaStream_t s)
{
    static_assert(L_STAGING_FITS<BN, SLOTS, BPRE, KB>, "the ring holds the TMA-store staging");
    using L = FusedLayout<BN, SLOTS, BPRE, KB>;
    auto kern = tc_fused_kernel<BN, SLOTS, BPRE, KB>;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = smem_limit_once(kern, L::SMEM_BYTES, smem_set); e != cudaSuccess) return e;
    const int work = a.dp_tiles + a.split_tiles * a.splits;
    const int grid = work < st.num_sms ? work : st.num_sms;
    if ((a.cluster > 1 && !L::CLUSTER_OK) || (a.fixup && !L::FIXUP_OK)) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3(grid), dim3(kFusedThreads), L::SMEM_BYTES, s, a.cluster, ta, tb, tbhi, tblo,
                      *reinterpret_cast<const CUtensorMap*>(st.tmap_c),
                      *reinterpret_cast<const CUtensorMap*>(st.tmap_p), a);
}

}  // namespace

cudaError_t tc_fused_main(int bn, int bk, bool b_presplit, const TcPlanState& st, const TcArgs& a,
                          const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbhi,
                          const CUtensorMap& tblo, cudaStream_t s)
{
    if (b_presplit) {
        switch (bn) {
        case 128: return launch_fused<128, 3, true, 32>(st, a, ta, tb, tbhi, tblo, s);
        case 256: return launch_fused<256, 2, true, 32>(st, a, ta, tb, tbhi, tblo, s);
        default: return cudaErrorInvalidValue;
        }
    }
    if (bk == 16) {
        switch (bn) {
        case 128: return launch_fused<128, 6, false, 16>(st, a, ta, tb, tbhi, tblo, s);
        case 256: return launch_fused<256, 4, false, 16>(st, a, ta, tb, tbhi, tblo, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
    case 128: return launch_fused<128, 3, false, 32>(st, a, ta, tb, tbhi, tblo, s);
    case 256: return launch_fused<256, 2, false, 32>(st, a, ta, tb, tbhi, tblo, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gemm_f32
