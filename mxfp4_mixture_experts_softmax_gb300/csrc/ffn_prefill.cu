// ffn_prefill.cu -- large-M grouped MXFP4 GEMMs on the 5th-generation tensor
// cores (tcgen05 MMA, accumulators in tensor memory).
//
// Prefill chunks put tens to thousands of rows on each expert, so the GEMMs
// become dense contractions (separate large-M launcher regime: vLLM MiniMax M3
// on MI355X, section "local shape and tiling"; padded and tuned prefill GEMM:
// VibeSys Qwen3.5-397B on 4x MI300A, section "baseline").
//
// Work item = one tile of N = tile_m token rows of one expert x one block of
// 128 weight rows (swap-AB: weights are the MMA's M = 128 side, tokens its N
// side).  Persistent CTAs (one per SM) loop over the items; warp roles:
//   * producer warp: 2D TMA loads of the block's packed codes (64 k per
//     stage, prefetched into L2 ahead of the ring) and of the tile's token
//     rows as one box in the 128-byte swizzled K-major layout the MMA reads
//     (gate_up reads x gathered into tile order by gather_rows_f16_kernel, down
//     reads h, which is already in tile order); both are f16 rows scaled per
//     row by a power of two (rows_to_f16_kernel), the factor undone in the
//     epilogue;
//   * 16 converter warps, four per tensor-memory lane quadrant, each owning
//     every fourth stage for its quadrant's 32 weight rows: dequantisation of
//     the codes by the hardware E2M1 -> f16x2 conversion and one f16x2
//     multiply by 2^(s - s_ref) (s_ref = max(s) - 13 over the weight row, so
//     the row fits f16, largest 6 * 2^13, and every group within 2^36 of the
//     row's largest scale stays exact; 2^(s_ref - 127) is applied per row in
//     the epilogue), written straight into the stage's A operand in tensor
//     memory (tcgen05.st; row = lane), so A never passes through shared
//     memory, whose bandwidth the B operand and the TMA writes need;
//   * MMA warp: one thread issues the four K = 16 tcgen05.mma of each stage
//     (A from tensor memory, B from shared memory) into the item's
//     accumulator and commits them to the stage's mbarrier, which frees the
//     stage (its shared-memory slot and its tensor-memory A columns);
//   * 4 epilogue warps: read the finished accumulator (each warp its 32
//     lanes), apply SwiGLU (gate and up rows interleaved, partner one lane
//     away) or the routing weight, and store; the accumulator is double
//     buffered (single for 256-wide tiles, for lack of tensor memory) so this
//     overlaps the next item's MMAs.
// Every wait is bounded (see mbar_wait); after a timeout each role stops, the
// MMA thread drains its own MMAs (bounded), and tensor memory is freed.
#include <stdlib.h>

#include <algorithm>

#include "moe_internal.h"
#include "tcgen05.cuh"

namespace moe {

namespace {

constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kConvWarp0 = 2;
constexpr int kConvWarps = 16;
constexpr int kEpiWarp0 = kConvWarp0 + kConvWarps;  // 18..21: warp % 4 covers every lane quadrant
constexpr int kEpiWarps = 4;
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;  // 704
constexpr int kBK = 64;                                   // k per stage (one 128-byte f16 row)
constexpr int kACols = kBK / 2;                           // tensor-memory columns of one A stage
constexpr int kCodeBytes = 128 * (kBK / 2);               // 4 KB packed codes stage
constexpr int kCodeBox = 64;                              // rows per codes box

// Instruction descriptor: f16 x f16 -> fp32 (a and b format fields 0), both
// operands K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) += A (tensor memory) * B (shared memory descriptor).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The pair form, issued by the even CTA of a CTA pair: M = 256, A rows 0..127
// from this CTA's tensor memory and 128..255 from the other CTA's at the same
// address, B's N rows split between the two CTAs' shared memory at the same
// offset (rows 0..N/2-1 here), D rows likewise split by CTA.
__device__ __forceinline__ void mma_f16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 consecutive 32-bit tensor-memory columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}


// Largest E8M0 byte of a weight row's K/32 scales, read by `parts` threads
// (part = 0..parts-1) that each take every parts-th 16-byte chunk (vec) or
// byte; the caller combines the parts.
__device__ __forceinline__ uint32_t row_scale_max_part(const uint8_t* sp, int ngroups, bool vec,
                                                       int part, int parts) {
    uint32_t m = 0;
    if (vec) {
        for (int c = part; c < ngroups / 16; c += parts) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(sp) + c);
            m = __vmaxu4(m, __vmaxu4(__vmaxu4(v.x, v.y), __vmaxu4(v.z, v.w)));
        }
        m = __vmaxu4(m, m >> 16);
        m = __vmaxu4(m, m >> 8);
        return m & 0xFFu;
    }
    for (int i = part; i < ngroups; i += parts) m = max(m, (uint32_t)__ldg(sp + i));
    return m;
}

// The row's reference exponent: its values are stored as f16 times 2^(s -
// s_ref), at most 6 * 2^13.
__device__ __forceinline__ int row_scale_ref(uint32_t smax) { return max((int)smax - 13, 1); }

// f16x2 (2^e, 2^e) for the group scale s: e = s - s_ref <= 13; below 2^-24 it
// rounds to zero (groups more than 2^36 under the row's largest).
__device__ __forceinline__ uint32_t f16_group_mult(uint32_t s, int s_ref) {
    const int e = min(max((int)s - s_ref, -30), 13);
    const __half h = __float2half_rn(__uint_as_float((uint32_t)(e + 127) << 23));
    return (uint32_t)__half_as_ushort(h) * 0x00010001u;
}

// Eight codes (two per byte, the even k in the low nibble) -> four f16x2
// (k0,k1), (k2,k3), (k4,k5), (k6,k7), each multiplied by `mult`.
__device__ __forceinline__ uint4 codes_to_f16x8(uint32_t w, uint32_t mult) {
    uint32_t r0, r1, r2, r3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(w));
    uint4 v;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(v.x) : "r"(r0), "r"(mult));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(v.y) : "r"(r1), "r"(mult));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(v.z) : "r"(r2), "r"(mult));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(v.w) : "r"(r3), "r"(mult));
    return v;
}

template <int N, bool PAIR>
struct PrefillSmem {
    // 128-row weight blocks per work item and CTA.  The blocks share the
    // tile's B stage, so B crosses L2 once per kRB blocks (the f16 B rows,
    // N * 128 bytes per 64-k stage against 4 KB of codes, make L2 ->
    // shared-memory traffic a bound).  Two blocks only where both
    // accumulators can still be double-buffered: at N = 128 the single buffer
    // and the 4-slot ring cost more than the saved traffic (skewed 8192
    // prefill 3.1 -> 3.8 ms; 1536-token prefill with N = 64: 1.86 -> 1.74 ms).
    // A CTA pair (PAIR) shares B instead: each CTA holds one block and loads
    // half of the tile's B rows, and one pair MMA (M = 256) reads both halves.
    static constexpr int kRB = (!PAIR && N <= 64) ? 2 : 1;
    static constexpr int kBRows = PAIR ? N / 2 : N;                // B rows this CTA loads
    static constexpr int kBBytes = kBRows * kBK * 2;
    static constexpr int kCodeStage = kRB * kCodeBytes;            // codes of the CTA's blocks
    static constexpr int kStage = kBBytes + kCodeStage;            // multiple of 1024
    static_assert(kStage % 1024 == 0, "swizzle atoms");
    // Converter warp (quadrant, part) owns the stages with gs % 4 == part; with
    // a ring of a multiple of 4 slots each slot belongs to one part, so every
    // barrier's phases are observed in order (a parity wait is unambiguous
    // only one phase ahead).
    // Two rings: kStages shared-memory slots (codes + B, filled by TMA) and
    // kAStages tensor-memory A slots (filled by the converters).  With two
    // blocks per item tensor memory holds only 4 A slots, but shared memory
    // holds 8 stages, so TMA runs further ahead than the conversion.
    // a pair's stages (half the B rows, no second block) are small enough
    // for 16 slots at 128-row tiles: 2.77 -> 2.71 ms on the skewed 8192-token
    // prefill; the A slots in tensor memory stay 8 (the rings decouple)
    static constexpr int kStages = (PAIR && 16 * kStage <= 200 * 1024) ? 16
                                   : 8 * kStage <= 170 * 1024       ? 8
                                                                    : 4;
    static constexpr int kAStages = (kRB == 1 && N <= 128) ? 8 : 4;
    static_assert(kStages % 4 == 0 && kAStages % 4 == 0, "slot ownership");
    static_assert(kStages % kAStages == 0, "ring nesting");
    static constexpr int kBars = kStages * kStage;
    static constexpr int kTotal = kBars + 256 + 1024;              // + alignment slack
    // tensor memory (512 columns): the accumulators (one per block, N
    // columns each), then the A stages (kACols columns per block)
    static constexpr int kAColsStage = kRB * kACols;
    static constexpr int kAccCols = kRB * N;
    static constexpr int kAccBufs = 2 * kAccCols + kAStages * kAColsStage <= 512 ? 2 : 1;
    static constexpr int kACol0 = kAccBufs * kAccCols;
    static_assert(kACol0 + kAStages * kAColsStage <= 512, "tensor memory");
};

template <int MODE, int N>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_gemm_kernel(const GroupedGemm g, const __grid_constant__ CUtensorMap codes_map,
                        const __grid_constant__ CUtensorMap act_map) {
    pdl_begin();
    using L = PrefillSmem<N, false>;
    constexpr int kStages = L::kStages, kAStages = L::kAStages;
    constexpr bool kDecoupled = kAStages != kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // The MMA thread waits and commits once per pair of stages (stages 2P and
    // 2P + 1 share pair barrier P mod kPairs): its per-stage barrier work,
    // not the tensor pipe, bounds the loop otherwise.
    constexpr int kPairs = kStages / 2, kAPairs = kAStages / 2;
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + L::kBars);  // codes + B landed, per slot
    uint64_t* a_full = raw_full + kStages;                               // A converted, per A pair
    uint64_t* stage_free = a_full + kAPairs;                             // MMAs done with a slot pair
    uint64_t* a_free = stage_free + kPairs;                              // MMAs done with an A pair
    uint64_t* acc_full = a_free + kAPairs;                               // [2] accumulator ready
    uint64_t* acc_free = acc_full + 2;                                   // [2] accumulator drained
    uint64_t* drain = acc_free + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    constexpr int kAccBufs = L::kAccBufs;
    auto stage_b = [&](int s) { return smem + s * L::kStage; };
    auto stage_c = [&](int s) { return smem + s * L::kStage + L::kBBytes; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = g.K;
    // stages per item, rounded up to whole pairs (a padding stage reads zero codes)
    const int nk = ((K + kBK - 1) / kBK + 1) & ~1;
    // blocks of 64 i (gate_up: 64 gate + 64 up rows) or of 128 rows (down);
    // an item is one tile x kRB consecutive blocks
    constexpr int kRB = L::kRB;
    const int row_blocks = MODE == 0 ? (g.I + 63) / 64 : (g.rows + 127) / 128;
    const int row_groups = (row_blocks + kRB - 1) / kRB;
    const int items = checked_tiles(g) * row_groups;
    constexpr uint32_t kTmemCols = 512;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&raw_full[s], 1);
        for (int p = 0; p < kPairs; ++p) mbar_init(&stage_free[p], 1);
        for (int p = 0; p < kAPairs; ++p) {
            mbar_init(&a_full[p], 8);  // one converter warp per lane quadrant and stage
            mbar_init(&a_free[p], 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_free[b], kEpiWarps);
        }
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------- producer
        uint32_t gs = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
            const int tile = item / row_groups, grp = item % row_groups;
            const int e = checked_expert(g, tile, grp == 0);
            if (e < 0) continue;  // skipped by every role
            // two 64-row code boxes per block: gate and up rows, or the
            // block's two halves
            int crow[2 * kRB];
#pragma unroll
            for (int j = 0; j < kRB; ++j) {
                const int block = grp * kRB + j;
                crow[2 * j] = e * g.rows + (MODE == 0 ? block * 64 : block * 128);
                crow[2 * j + 1] = MODE == 0 ? e * g.rows + g.I + block * 64 : crow[2 * j] + kCodeBox;
            }
            // no L2 prefetches ahead of the ring (1536-token prefill: 1.62 -> 1.57 ms
            // without them)
            for (int st = 0; st < nk; ++st, ++gs) {
                const int s = gs % kStages;
                // both slots of a pair come free with the pair's commit
                if (gs >= kStages && (gs & 1) == 0 &&
                    !mbar_wait_warp(&stage_free[(gs >> 1) % kPairs], ((gs / kStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&raw_full[s], (uint32_t)(L::kCodeStage + L::kBBytes));
#pragma unroll
                    for (int j = 0; j < kRB; ++j) {
                        const uint32_t cdst = smem_u32(stage_c(s)) + j * kCodeBytes;
                        tma_load_2d(cdst, &codes_map, st * (kBK / 2), crow[2 * j], &raw_full[s]);
                        tma_load_2d(cdst + kCodeBox * (kBK / 2), &codes_map, st * (kBK / 2),
                                    crow[2 * j + 1], &raw_full[s]);
                    }
                    tma_load_2d(smem_u32(stage_b(s)), &act_map, st * kBK, tile * N, &raw_full[s]);
                }
            }
        }
        // wait (bounded) until the last loads landed before the CTA can exit
        if (lane == 0)
            for (int d = 0; d < kStages && d < (int)gs; ++d) {
                const uint32_t u = gs - 1 - d;
                if (!mbar_wait(&raw_full[u % kStages], (u / kStages) & 1)) break;
            }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(128, N);
            uint32_t gs = 0, it = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
                if (checked_expert(g, item / row_groups, false) < 0) continue;
                const uint32_t b = it % kAccBufs;
                if (it >= (uint32_t)kAccBufs && !mbar_wait(&acc_free[b], ((it / kAccBufs) - 1) & 1)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + b * L::kAccCols;
                for (int st = 0; st < nk; st += 2, gs += 2) {
                    const int pr = (gs >> 1) % kPairs, pa = (gs >> 1) % kAPairs;
                    // both stages' A converted; the converters arrive only after
                    // seeing their stage's TMA barrier, so B has landed too
                    if (!mbar_wait(&a_full[pa], (gs / kAStages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int s = (gs + h2) % kStages, sa = (gs + h2) % kAStages;
                        const uint64_t bd = sdesc_sw128(smem_u32(stage_b(s)));
#pragma unroll
                        for (int j = 0; j < kRB; ++j) {  // each block into its own accumulator
                            const uint32_t a_tmem =
                                tmem + (uint32_t)(L::kACol0 + sa * L::kAColsStage + j * kACols);
#pragma unroll
                            for (int k = 0; k < kBK / 16; ++k)  // A: 8 columns per K = 16; B: +32 bytes in the swizzle atom
                                mma_f16_ts(d_tmem + (uint32_t)(j * N), a_tmem + 8u * k, bd + 2u * k,
                                           idesc, (st | h2 | k) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(&stage_free[pr]);
                    if (kDecoupled) mma_commit(&a_free[pa]);
                }
                if (ok) mma_commit(&acc_full[b]);
                ++it;  // items processed (skipped ones use no accumulator)
            }
            mma_commit(drain);  // every MMA this thread issued has completed when this arrives
            mbar_wait(drain, 0);
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------ converters
        // warp w serves lane quadrant w % 4 (the tensor-memory lanes it may
        // write) and owns the stages with gs % 4 == (w - kConvWarp0) / 4
        const int quad = warp & 3, part = (warp - kConvWarp0) >> 2;
        const int rho = 32 * quad + lane;  // A row = tensor-memory lane
        const int crow = MODE == 0 ? ((rho & 1) ? kCodeBox + (rho >> 1) : rho >> 1) : rho;
        const bool svec = (K % 512) == 0 && ((reinterpret_cast<uintptr_t>(g.scales) & 15) == 0);
        const int ngroups = K / 32;
        const bool s2 = (ngroups % 2) == 0 && ((reinterpret_cast<uintptr_t>(g.scales) & 1) == 0);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)L::kACol0;
        uint32_t gs = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
            const int tile = item / row_groups, grp = item % row_groups;
            const int e = checked_expert(g, tile, false);
            if (e < 0) continue;
            // this lane's weight row in each of the item's blocks
            const uint8_t* sp[kRB];
            int s_ref[kRB];
            bool rvalid[kRB];
#pragma unroll
            for (int j = 0; j < kRB; ++j) {
                const int block = grp * kRB + j;
                int wrow;
                if (MODE == 0) {
                    const int n = block * 64 + (rho >> 1);
                    rvalid[j] = n < g.I;
                    wrow = (rho & 1) ? g.I + n : n;
                } else {
                    wrow = block * 128 + rho;
                    rvalid[j] = wrow < g.rows;
                }
                sp[j] = g.scales + ((size_t)e * g.rows + (rvalid[j] ? wrow : 0)) * (size_t)ngroups;
                s_ref[j] = row_scale_ref(rvalid[j] ? row_scale_max_part(sp[j], ngroups, svec, 0, 1) : 0u);
            }
            // the stage's two scale groups of a row (bytes 2st, 2st + 1): one
            // 16-bit load where aligned (a 32-sector load per warp either way,
            // so one load instead of two halves the L1 wavefronts)
            auto scales2 = [&](int j, int st) -> uint32_t {
                if (!rvalid[j]) return 0u;
                if (s2 && 2 * st + 1 < ngroups)
                    return (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(sp[j]) + st);
                uint32_t v = 0;
                if (2 * st < ngroups) v = (uint32_t)__ldg(sp[j] + 2 * st);
                if (2 * st + 1 < ngroups) v |= (uint32_t)__ldg(sp[j] + 2 * st + 1) << 8;
                return v;
            };
            for (int st = 0; st < nk; ++st, ++gs) {
                if ((int)(gs & 3u) != part) continue;
                const int s = gs % kStages, sa = gs % kAStages;
                uint32_t m0[kRB], m1[kRB];
#pragma unroll
                for (int j = 0; j < kRB; ++j) {
                    const uint32_t sc = scales2(j, st);
                    m0[j] = f16_group_mult(sc & 0xFFu, s_ref[j]);
                    m1[j] = f16_group_mult(sc >> 8, s_ref[j]);
                }
                if (!mbar_wait_warp(&raw_full[s], (gs / kStages) & 1)) {
                    ok = false;
                    break;
                }
                // the A slot comes free with the MMAs of stage gs - kAStages (with
                // equal rings the TMA barrier already implies it)
                if (kDecoupled && gs >= (uint32_t)kAStages &&
                    !mbar_wait_warp(&a_free[(gs >> 1) % kAPairs], ((gs / kAStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();  // after the MMAs that last read this A stage
#pragma unroll
                for (int j = 0; j < kRB; ++j) {
                    uint4 c[2];
                    const uint32_t cs = smem_u32(stage_c(s)) + j * kCodeBytes + crow * (kBK / 2);
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(c[0].x), "=r"(c[0].y), "=r"(c[0].z), "=r"(c[0].w)
                                 : "r"(cs));
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(c[1].x), "=r"(c[1].y), "=r"(c[1].z), "=r"(c[1].w)
                                 : "r"(cs + 16));
                    uint32_t a[32];  // column i of the block's stage = f16x2 (k 2i, 2i + 1)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t w[4] = {c[hh].x, c[hh].y, c[hh].z, c[hh].w};
                        const uint32_t m = hh ? m1[j] : m0[j];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint4 v = codes_to_f16x8(w[i], m);
                            a[16 * hh + 4 * i + 0] = v.x;
                            a[16 * hh + 4 * i + 1] = v.y;
                            a[16 * hh + 4 * i + 2] = v.z;
                            a[16 * hh + 4 * i + 3] = v.w;
                        }
                    }
                    tmem_st32(lane_base + (uint32_t)(sa * L::kAColsStage + j * kACols), a);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[(gs >> 1) % kAPairs]);
            }
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int quad = warp & 3;  // tensor-memory lanes 32*quad .. 32*quad + 31
        const int r = 32 * quad + lane;
        const bool svec = (K % 512) == 0 && ((reinterpret_cast<uintptr_t>(g.scales) & 15) == 0);
        // Per item: this lane's weight row factor 2^(s_ref - 127) (the part of
        // the scales the converters left out; accumulator lane r holds A row
        // r) and the tile's pair indices and column factors (column j in lane
        // j % 32 of register j / 32; the factor undoes the B row's scaling,
        // per token for x, per position for h, and in the down GEMM includes
        // the routing weight).  Loaded one item ahead: frn, qn, cn hold the
        // values of `item` at the top of the loop.
        constexpr int kQ = N / 32;
        int qn[kQ];
        float cn[kQ];
        float frn[kRB];
        auto load_item = [&](int item) {
            if (item >= items) return;
            const int tile = item / row_groups, grp = item % row_groups;
            const int e = checked_expert(g, tile, false);
            if (e < 0) return;
#pragma unroll
            for (int j = 0; j < kRB; ++j) {
                const int block = grp * kRB + j;
                int wrow;
                bool rvalid;
                if (MODE == 0) {
                    const int n = block * 64 + (r >> 1);
                    rvalid = n < g.I;
                    wrow = (r & 1) ? g.I + n : n;
                } else {
                    wrow = block * 128 + r;
                    rvalid = wrow < g.rows;
                }
                const uint8_t* sp = g.scales + ((size_t)e * g.rows + (rvalid ? wrow : 0)) * (size_t)(K / 32);
                frn[j] = __uint_as_float(
                    (uint32_t)row_scale_ref(rvalid ? row_scale_max_part(sp, K / 32, svec, 0, 1) : 0u) << 23);
            }
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                const int p = tile * N + 32 * u + lane;
                qn[u] = checked_pair(g, p);
                if (MODE == 0)
                    cn[u] = qn[u] < 0 ? 0.0f : __ldg(g.act_rscale + qn[u] / g.Kt);
                else if (!g.y_blocked)  // blocked y leaves the column factor to the combine
                    cn[u] = qn[u] < 0 ? 0.0f : __ldg(g.topk_w + qn[u]) * __ldg(g.act_rscale + p);
                else
                    cn[u] = 0.0f;
            }
        };
        load_item(blockIdx.x);
        uint32_t it = 0;
        for (int item = blockIdx.x; item < items; item += gridDim.x) {
            const int tile = item / row_groups, grp = item % row_groups;
            const int e = checked_expert(g, tile, false);
            if (e < 0) {
                load_item(item + gridDim.x);
                continue;
            }
            const uint32_t b = it % kAccBufs;
            float frs[kRB];
#pragma unroll
            for (int j = 0; j < kRB; ++j) frs[j] = frn[j];
            int qv[kQ];
            float cv[kQ];
#pragma unroll
            for (int u = 0; u < kQ; ++u) qv[u] = qn[u], cv[u] = cn[u];
            // positions holding a pair: a prefix of the tile (padding follows
            // an expert's pairs)
            int nvalid = 0;
            if (MODE == 1) {
#pragma unroll
                for (int u = 0; u < kQ; ++u) nvalid += __popc(__ballot_sync(0xFFFFFFFFu, qv[u] >= 0));
            }
            if (!mbar_wait_warp(&acc_full[b], (it / kAccBufs) & 1)) break;
            tc_fence_after();
            load_item(item + gridDim.x);
            // 32 columns per round trip: two loads, one wait; block by block
            // (not unrolled across blocks: that doubles the live registers)
#pragma unroll 1
            for (int j = 0; j < kRB; ++j) {
            const int block = grp * kRB + j;
            const float fr = j == 0 ? frs[0] : frs[kRB - 1];
#pragma unroll
            for (int c0 = 0; c0 < N; c0 += 32) {
                uint32_t v[32];
                const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16) + b * L::kAccCols +
                                       (uint32_t)(j * N + c0);
                tmem_ld16_nowait(taddr, v);
                tmem_ld16_nowait(taddr + 16, v + 16);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                const int q_lo = qv[c0 / 32];
                const float c_lo = cv[c0 / 32];
                if (MODE == 0) {
                    // lane 2i holds gate row i, lane 2i+1 up row i: after one
                    // exchange per column pair the even lane owns column j and
                    // the odd lane column j + 1
                    const int n = block * 64 + (r >> 1);
                    const bool odd = lane & 1;
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float a0 = __uint_as_float(v[i]) * fr, a1 = __uint_as_float(v[i + 1]) * fr;
                        const float other = __shfl_xor_sync(0xFFFFFFFFu, odd ? a0 : a1, 1);
                        const int j = c0 + i + (odd ? 1 : 0);
                        const float gate = odd ? other : a0;   // even: own gate j; odd: partner's gate j+1
                        const float up = odd ? a1 : other;     // even: partner's up j; odd: own up j+1
                        const int q = __shfl_sync(0xFFFFFFFFu, q_lo, j & 31);
                        const float fc = __shfl_sync(0xFFFFFFFFu, c_lo, j & 31);
                        if (n < g.I && q >= 0)
                            g.h_out[(size_t)(tile * N + j) * g.I + n] =
                                f32_to_bf16_bits(silu(gate * fc) * (up * fc));
                    }
                } else if (g.y_blocked) {
                    // y staged as scaled f16 rows by position, written for the
                    // positions holding a pair; the column factor (routing
                    // weight x h row factor) is applied by the combine
                    const int m = block * 128 + r;
                    const int nc = nvalid - c0;  // warp-uniform
                    store_y16_chunk(g, v, fr, block, quad, lane, tile * N + c0, nc, m < g.rows);
                } else {  // y[pair][m]
                    const int m = block * 128 + r;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int q = __shfl_sync(0xFFFFFFFFu, q_lo, i);
                        const float fc = __shfl_sync(0xFFFFFFFFu, c_lo, i);
                        if (m < g.rows && q >= 0)
                            g.y_out[(size_t)q * g.rows + m] = fc * (__uint_as_float(v[i]) * fr);
                    }
                }
            }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_free[b]);
            ++it;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
    pdl_end();
}

// The CTA-pair form of the kernel above (launched as clusters of 2): a work
// item is one tile x two adjacent 128-row weight blocks, block 2 grp + rank
// in CTA `rank` of the pair.  Each CTA loads its block's codes and half of the
// tile's B rows (N / 2 rows, at the same shared-memory offset in both CTAs)
// and converts its block into its own tensor memory; the even CTA's MMA
// thread issues one M = 256 MMA per K = 16 for both (tcgen05 cta_group::2),
// which reads both CTAs' A and B halves, and commits to the barriers of both
// CTAs.  B crosses L2 -> shared memory once per 256 weight rows instead of
// once per 128.  The odd CTA's converter and epilogue warps arrive on the
// even CTA's barriers; its MMA warp only allocates and frees tensor memory.
template <int MODE, int N>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const GroupedGemm g, const __grid_constant__ CUtensorMap codes_map,
                        const __grid_constant__ CUtensorMap act_map) {
    pdl_begin();
    using L = PrefillSmem<N, true>;
    constexpr int kStages = L::kStages, kAStages = L::kAStages;
    constexpr bool kDecoupled = kAStages != kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // The MMA thread waits on the converters once per group of four stages
    // and releases the group's slots with one commit: each wait and commit
    // costs the issuing thread about as much as two MMAs.
    constexpr int kAPairs = kAStages / 2;
    constexpr int kGroups = kStages / 4, kAGroups = kAStages / 4;
    static_assert(kStages % 4 == 0 && kAStages % 4 == 0, "groups of four stages");
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + L::kBars);  // codes + B landed, per slot
    uint64_t* a_full = raw_full + kStages;      // A converted in both CTAs, per A pair (even CTA)
    // MMAs of a group of four stages completed: frees the group's shared-
    // memory slots (waited by the producer, kGroups groups later) and its A
    // slots (waited by the converters, kAGroups groups later) with one commit
    uint64_t* grp_done = a_full + kAPairs;
    uint64_t* acc_full = grp_done + kGroups;    // [2] accumulator ready
    uint64_t* acc_free = acc_full + 2;          // [2] drained by both CTAs (even CTA)
    uint64_t* drain = acc_free + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    constexpr int kAccBufs = L::kAccBufs;
    auto stage_b = [&](int s) { return smem + s * L::kStage; };
    auto stage_c = [&](int s) { return smem + s * L::kStage + L::kBBytes; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // clusters of 2 along x: the rank in the pair is the low bit of the CTA index
    const int rank = (int)(blockIdx.x & 1u);
    const int K = g.K;
    const int nk = ((K + kBK - 1) / kBK + 3) & ~3;  // stages per item, whole groups of four
    const int row_blocks = MODE == 0 ? (g.I + 63) / 64 : (g.rows + 127) / 128;
    const int row_groups = row_blocks / 2;          // even (checked by the launcher)
    const int items = checked_tiles(g) * row_groups;
    constexpr uint32_t kTmemCols = 512;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&raw_full[s], 1);
        for (int p = 0; p < kGroups; ++p) mbar_init(&grp_done[p], 1);
        for (int p = 0; p < kAGroups; ++p)
            mbar_init(&a_full[p], 16);  // per stage pair one converter warp per lane quadrant: 2 pairs, 2 CTAs
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_free[b], 2 * kEpiWarps);
        }
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) tmem_alloc<true>(tmem_slot, kTmemCols);
    tc_fence_before();
    // the other CTA's barriers are initialised and its tensor memory
    // allocated before anything arrives there or an MMA writes it
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------- producer
        uint32_t gs = 0;
        bool ok = true;
        for (int item = blockIdx.x >> 1; item < items && ok; item += gridDim.x >> 1) {
            const int tile = item / row_groups, block = 2 * (item % row_groups) + rank;
            const int e = checked_expert(g, tile, block == 0);
            if (e < 0) continue;  // skipped by every role of both CTAs
            const int crow0 = e * g.rows + (MODE == 0 ? block * 64 : block * 128);
            const int crow1 = MODE == 0 ? e * g.rows + g.I + block * 64 : crow0 + kCodeBox;
            const int brow = tile * N + rank * L::kBRows;
            // no L2 prefetches ahead of the ring: on the skewed 8192-token
            // prefill they cost 11% of the layer (3.11 -> 2.77 ms without)
            for (int st = 0; st < nk; ++st, ++gs) {
                const int s = gs % kStages;
                // four slots come free with their group's commit
                if (gs >= kStages && (gs & 3) == 0 &&
                    !mbar_wait_warp(&grp_done[(gs >> 2) % kGroups], ((gs / kStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&raw_full[s], (uint32_t)(L::kCodeStage + L::kBBytes));
                    const uint32_t cdst = smem_u32(stage_c(s));
                    tma_load_2d(cdst, &codes_map, st * (kBK / 2), crow0, &raw_full[s]);
                    tma_load_2d(cdst + kCodeBox * (kBK / 2), &codes_map, st * (kBK / 2), crow1,
                                &raw_full[s]);
                    tma_load_2d(smem_u32(stage_b(s)), &act_map, st * kBK, brow, &raw_full[s]);
                }
            }
        }
        if (lane == 0)  // the last loads landed before the CTA can exit (bounded)
            for (int d = 0; d < kStages && d < (int)gs; ++d) {
                const uint32_t u = gs - 1 - d;
                if (!mbar_wait(&raw_full[u % kStages], (u / kStages) & 1)) break;
            }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_f16(256, N);
            uint32_t gs = 0, it = 0;
            bool ok = true;
            for (int item = blockIdx.x >> 1; item < items && ok; item += gridDim.x >> 1) {
                if (checked_expert(g, item / row_groups, false) < 0) continue;
                const uint32_t b = it % kAccBufs;
                if (it >= (uint32_t)kAccBufs && !mbar_wait(&acc_free[b], ((it / kAccBufs) - 1) & 1)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + b * L::kAccCols;
                for (int st = 0; st < nk; st += 4, gs += 4) {
                    // the group's four stages converted in both CTAs (the
                    // converters arrive after their stage's TMA barrier: B has
                    // landed)
                    if (!mbar_wait(&a_full[(gs >> 2) % kAGroups], (gs / kAStages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2) {
                        const int s = (gs + h2) % kStages, sa = (gs + h2) % kAStages;
                        const uint64_t bd = sdesc_sw128(smem_u32(stage_b(s)));
                        const uint32_t a_tmem = tmem + (uint32_t)(L::kACol0 + sa * kACols);
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k)
                            mma_f16_ts_pair(d_tmem, a_tmem + 8u * k, bd + 2u * k, idesc,
                                            (st | h2 | k) != 0 ? 1u : 0u);
                    }
                    mma_commit_pair(&grp_done[(gs >> 2) % kGroups]);  // release the group's slots
                }
                if (ok) mma_commit_pair(&acc_full[b]);
                ++it;
            }
            mma_commit_pair(drain);  // both CTAs: every MMA of the pair has completed
            mbar_wait(drain, 0);
        } else if (lane == 0) {
            // the odd CTA: the pair's MMAs, and the commits arriving on this
            // CTA's barriers as they complete, are done before it exits
            mbar_wait(drain, 0);
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------ converters
        // warp (quadrant, part) converts its quadrant's 32 weight rows for the
        // stage pairs P (stages 2P, 2P + 1, counted over all items) with
        // P % kParts == part; the pair's four scale groups of a row are one
        // 32-bit load.  kParts = the A-slot pairs (at most 4): every slot, its
        // TMA barrier and its A-slot barrier then belong to one part, which
        // waits on each of their phases in order (a parity wait is unambiguous
        // only one phase ahead).  With 4 A slots (256-row tiles) half the
        // converter warps stay idle; the MMAs take twice as long per stage.
        constexpr int kParts = kAPairs < 4 ? kAPairs : 4;
        static_assert((kStages / 2) % kParts == 0, "slot ownership");
        const int quad = warp & 3, part = (warp - kConvWarp0) >> 2;
        const int rho = 32 * quad + lane;
        const int crow = MODE == 0 ? ((rho & 1) ? kCodeBox + (rho >> 1) : rho >> 1) : rho;
        const bool svec = (K % 512) == 0 && ((reinterpret_cast<uintptr_t>(g.scales) & 15) == 0);
        const int ngroups = K / 32;
        const bool s4 = (ngroups % 4) == 0 && ((reinterpret_cast<uintptr_t>(g.scales) & 3) == 0);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)L::kACol0;
        uint32_t gs = 0;  // the item's first stage, counted over all items (even)
        bool ok = true;
        for (int item = blockIdx.x >> 1; item < items && ok; item += gridDim.x >> 1) {
            const int tile = item / row_groups, block = 2 * (item % row_groups) + rank;
            const int e = checked_expert(g, tile, false);
            if (e < 0) continue;
            int wrow;
            bool rvalid;
            if (MODE == 0) {
                const int n = block * 64 + (rho >> 1);
                rvalid = n < g.I;
                wrow = (rho & 1) ? g.I + n : n;
            } else {
                wrow = block * 128 + rho;
                rvalid = wrow < g.rows;
            }
            const uint8_t* sp = g.scales + ((size_t)e * g.rows + (rvalid ? wrow : 0)) * (size_t)ngroups;
            const int s_ref = row_scale_ref(rvalid ? row_scale_max_part(sp, ngroups, svec, 0, 1) : 0u);
            // scale bytes of groups 4p .. 4p + 3 (stage pair p of the item), 0 past the row
            auto scales4 = [&](int p) -> uint32_t {
                if (!rvalid) return 0u;
                if (s4 && 4 * p + 3 < ngroups) return __ldg(reinterpret_cast<const uint32_t*>(sp) + p);
                uint32_t v = 0;
                for (int i = 0; i < 4; ++i)
                    if (4 * p + i < ngroups) v |= (uint32_t)__ldg(sp + 4 * p + i) << (8 * i);
                return v;
            };
            const int np = nk / 2;
            // this warp's first pair of the item (np when the part is idle)
            const int p0 = part < kParts
                               ? (part - (int)((gs >> 1) % (uint32_t)kParts) + kParts) % kParts
                               : np;
            uint32_t sc = p0 < np ? scales4(p0) : 0u;  // loaded one of this warp's pairs ahead
            for (int p = p0; p < np; p += kParts) {
                const uint32_t g0 = gs + 2u * (uint32_t)p;  // first stage of the pair
                const uint32_t scv = sc;
                if (p + kParts < np) sc = scales4(p + kParts);
                if (kDecoupled && g0 >= (uint32_t)kAStages &&
                    !mbar_wait_warp(&grp_done[((g0 >> 2) - kAGroups) % kGroups],
                                    (((g0 >> 2) - kAGroups) / kGroups) & 1)) {
                    ok = false;
                    break;
                }
#pragma unroll 1
                for (int h2 = 0; h2 < 2; ++h2) {
                    const uint32_t g_s = g0 + (uint32_t)h2;
                    const int s = g_s % kStages, sa = g_s % kAStages;
                    const uint32_t m0 = f16_group_mult((scv >> (16 * h2)) & 0xFFu, s_ref);
                    const uint32_t m1 = f16_group_mult((scv >> (16 * h2 + 8)) & 0xFFu, s_ref);
                    if (!mbar_wait_warp(&raw_full[s], (g_s / kStages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();  // after the MMAs that last read this A stage
                    uint4 c[2];
                    const uint32_t cs = smem_u32(stage_c(s)) + crow * (kBK / 2);
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(c[0].x), "=r"(c[0].y), "=r"(c[0].z), "=r"(c[0].w)
                                 : "r"(cs));
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(c[1].x), "=r"(c[1].y), "=r"(c[1].z), "=r"(c[1].w)
                                 : "r"(cs + 16));
                    uint32_t a[32];  // column i of the stage = f16x2 (k 2i, 2i + 1)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t w[4] = {c[hh].x, c[hh].y, c[hh].z, c[hh].w};
                        const uint32_t m = hh ? m1 : m0;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint4 v = codes_to_f16x8(w[i], m);
                            a[16 * hh + 4 * i + 0] = v.x;
                            a[16 * hh + 4 * i + 1] = v.y;
                            a[16 * hh + 4 * i + 2] = v.z;
                            a[16 * hh + 4 * i + 3] = v.w;
                        }
                    }
                    tmem_st32(lane_base + (uint32_t)(sa * kACols), a);
                }
                if (!ok) break;
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(&a_full[(g0 >> 2) % kAGroups], 0);
            }
            gs += (uint32_t)nk;
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int r = 32 * quad + lane;
        const bool svec = (K % 512) == 0 && ((reinterpret_cast<uintptr_t>(g.scales) & 15) == 0);
        constexpr int kQ = N / 32;
        int qn[kQ];
        float cn[kQ];
        float frn = 0.0f;
        auto load_item = [&](int item) {
            if (item >= items) return;
            const int tile = item / row_groups, block = 2 * (item % row_groups) + rank;
            const int e = checked_expert(g, tile, false);
            if (e < 0) return;
            int wrow;
            bool rvalid;
            if (MODE == 0) {
                const int n = block * 64 + (r >> 1);
                rvalid = n < g.I;
                wrow = (r & 1) ? g.I + n : n;
            } else {
                wrow = block * 128 + r;
                rvalid = wrow < g.rows;
            }
            const uint8_t* sp = g.scales + ((size_t)e * g.rows + (rvalid ? wrow : 0)) * (size_t)(K / 32);
            frn = __uint_as_float(
                (uint32_t)row_scale_ref(rvalid ? row_scale_max_part(sp, K / 32, svec, 0, 1) : 0u) << 23);
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                const int p = tile * N + 32 * u + lane;
                qn[u] = checked_pair(g, p);
                if (MODE == 0)
                    cn[u] = qn[u] < 0 ? 0.0f : __ldg(g.act_rscale + qn[u] / g.Kt);
                else if (!g.y_blocked)
                    cn[u] = qn[u] < 0 ? 0.0f : __ldg(g.topk_w + qn[u]) * __ldg(g.act_rscale + p);
                else
                    cn[u] = 0.0f;
            }
        };
        load_item(blockIdx.x >> 1);
        uint32_t it = 0;
        for (int item = blockIdx.x >> 1; item < items; item += gridDim.x >> 1) {
            const int tile = item / row_groups, block = 2 * (item % row_groups) + rank;
            const int e = checked_expert(g, tile, false);
            if (e < 0) {
                load_item(item + (gridDim.x >> 1));
                continue;
            }
            const uint32_t b = it % kAccBufs;
            const float fr = frn;
            int qv[kQ];
            float cv[kQ];
#pragma unroll
            for (int u = 0; u < kQ; ++u) qv[u] = qn[u], cv[u] = cn[u];
            int nvalid = 0;
            if (MODE == 1) {
#pragma unroll
                for (int u = 0; u < kQ; ++u) nvalid += __popc(__ballot_sync(0xFFFFFFFFu, qv[u] >= 0));
            }
            if (!mbar_wait_warp(&acc_full[b], (it / kAccBufs) & 1)) break;
            tc_fence_after();
            load_item(item + (gridDim.x >> 1));
#pragma unroll
            for (int c0 = 0; c0 < N; c0 += 32) {
                uint32_t v[32];
                const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16) + b * L::kAccCols + (uint32_t)c0;
                tmem_ld16_nowait(taddr, v);
                tmem_ld16_nowait(taddr + 16, v + 16);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                const int q_lo = qv[c0 / 32];
                const float c_lo = cv[c0 / 32];
                if (MODE == 0) {
                    const int n = block * 64 + (r >> 1);
                    const bool odd = lane & 1;
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float a0 = __uint_as_float(v[i]) * fr, a1 = __uint_as_float(v[i + 1]) * fr;
                        const float other = __shfl_xor_sync(0xFFFFFFFFu, odd ? a0 : a1, 1);
                        const int j = c0 + i + (odd ? 1 : 0);
                        const float gate = odd ? other : a0;
                        const float up = odd ? a1 : other;
                        const int q = __shfl_sync(0xFFFFFFFFu, q_lo, j & 31);
                        const float fc = __shfl_sync(0xFFFFFFFFu, c_lo, j & 31);
                        if (n < g.I && q >= 0)
                            g.h_out[(size_t)(tile * N + j) * g.I + n] =
                                f32_to_bf16_bits(silu_fast(gate * fc) * (up * fc));
                    }
                } else if (g.y_blocked) {
                    const int m = block * 128 + r;
                    const int nc = nvalid - c0;
                    store_y16_chunk(g, v, fr, block, quad, lane, tile * N + c0, nc, m < g.rows);
                } else {
                    const int m = block * 128 + r;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int q = __shfl_sync(0xFFFFFFFFu, q_lo, i);
                        const float fc = __shfl_sync(0xFFFFFFFFu, c_lo, i);
                        if (m < g.rows && q >= 0)
                            g.y_out[(size_t)q * g.rows + m] = fc * (__uint_as_float(v[i]) * fr);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(&acc_free[b], 0);  // the even CTA's MMA thread waits
            ++it;
        }
    }

    tc_fence_before();
    // neither CTA releases its tensor memory or shared memory while the other
    // may still arrive there or the pair's MMAs may still run
    cluster_sync_all();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc<true>(tmem, kTmemCols);
    }
    pdl_end();
}

template <int MODE, int N, bool PAIR>
cudaError_t launch_n(const GroupedGemm& g, cudaStream_t s) {
    using L = PrefillSmem<N, PAIR>;
    const size_t smem = L::kTotal;
    const void* fn;
    if constexpr (PAIR)
        fn = (const void*)prefill_pair_kernel<MODE, N>;
    else
        fn = (const void*)prefill_gemm_kernel<MODE, N>;
    cudaError_t err = ensure_dynamic_smem(fn, smem);
    if (err != cudaSuccess) return err;
    CUtensorMap codes_map, act_map;
    err = encode_2d_map(&codes_map, g.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.K / 2,
                        (uint64_t)g.num_experts * g.rows, g.K / 2, kBK / 2, kCodeBox,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    if (err != cudaSuccess) return err;
    // activations in tile order (gathered x for gate_up, h for down): the
    // CTA's B rows of a tile per box (all N, or its half of a pair's tile)
    err = encode_2d_map(&act_map, g.act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g.K, (uint64_t)g.act_rows,
                        (uint64_t)g.K * 2, kBK, L::kBRows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
    const int row_blocks = MODE == 0 ? (g.I + 63) / 64 : (g.rows + 127) / 128;
    const int row_groups = PAIR ? row_blocks / 2 : (row_blocks + L::kRB - 1) / L::kRB;
    const long long max_items = (long long)g.max_tiles * row_groups;
    if constexpr (PAIR) {
        // one wave of pairs: as many as can be resident at once (a pair needs
        // two SMs of one GPC), one item per pair at least
        int resident = 0;
        err = max_active_pairs(fn, kThreads, smem, &resident);
        if (err != cudaSuccess) return err;
        const int pairs = (int)std::min<long long>(max_items, (long long)std::max(resident, 1));
        return launch_pdl_cluster(prefill_pair_kernel<MODE, N>, dim3(2 * pairs),
                                  dim3(kThreads), smem, s, 2u, g, codes_map, act_map);
    } else {
        const int grid = (int)std::min<long long>(max_items, (long long)num_sms());
        return launch_pdl(prefill_gemm_kernel<MODE, N>, dim3(grid), dim3(kThreads), smem, s, g,
                          codes_map, act_map);
    }
}

// CTA pairs (two 128-row weight blocks sharing each B stage, one per CTA)
// for tiles of 128 or more rows whenever the blocks pair up evenly (with
// 64-row tiles the single-CTA kernel, two blocks per CTA, is faster);
// MOE_PREFILL_PAIR=0 selects the single-CTA kernel (for comparisons).
static bool use_pairs(const GroupedGemm& g, int mode) {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("MOE_PREFILL_PAIR");
        env = (v && v[0] == '0') ? 0 : 1;
    }
    const int row_blocks = mode == 0 ? (g.I + 63) / 64 : (g.rows + 127) / 128;
    return env == 1 && g.tile_m >= 128 && row_blocks % 2 == 0;
}

template <int MODE>
cudaError_t launch_mode(const GroupedGemm& g, cudaStream_t s) {
    if (g.max_tiles == 0) return cudaSuccess;
    const bool pair = use_pairs(g, MODE);
    switch (g.tile_m) {
        case 32: return launch_n<MODE, 32, false>(g, s);
        case 64: return pair ? launch_n<MODE, 64, true>(g, s) : launch_n<MODE, 64, false>(g, s);
        case 128: return pair ? launch_n<MODE, 128, true>(g, s) : launch_n<MODE, 128, false>(g, s);
        case 256: return pair ? launch_n<MODE, 256, true>(g, s) : launch_n<MODE, 256, false>(g, s);
        default: return cudaErrorInvalidValue;
    }
}

// xg[p] = f16(x[t] * 2^sigma_t), t the token of sorted position p's pair, for
// the rows of the used tiles (zero rows for padding), and rscale[t] =
// 2^-sigma_t: rows_to_f16_kernel's conversion of x applied while gathering
// into tile order, so x never exists as a separate f16 copy.  One warp per
// position (grid-stride).  Rows of up to 32 * NPL 16-byte pieces stay in
// registers (one pass over the token's bf16 row, read from L2); longer rows
// (NPL = 0) take a pass for the largest magnitude and one to convert.  The
// copy is written with streaming (evict-first) stores, so the far larger
// stream of gathered rows does not push x out of L2 while its Kt positions
// are read.  Every position of a token writes the same rscale value.
template <int NPL>
__global__ void __launch_bounds__(256) gather_rows_f16_kernel(const uint4* __restrict__ x, int H8,
                                                              const int32_t* __restrict__ sorted_pairs,
                                                              const int32_t* __restrict__ num_tiles,
                                                              int tile_m, int Kt, int cap, int num_pairs,
                                                              uint4* __restrict__ xg,
                                                              float* __restrict__ rscale) {
    pdl_begin();
    const int rows = min(max(__ldg(num_tiles), 0) * tile_m, cap);  // clamped like checked_tiles
    const int lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
    for (int p = blockIdx.x * wpb + (threadIdx.x >> 5); p < rows; p += gridDim.x * wpb) {
        int q = __ldg(sorted_pairs + p);
        if (q >= num_pairs) {
            if (lane == 0) flag_index_error();
            q = -1;
        }
        uint4* dst = xg + (size_t)p * H8;
        if (q < 0) {
            for (int c = lane; c < H8; c += 32) __stcs(dst + c, make_uint4(0, 0, 0, 0));
            continue;
        }
        const int t = q / Kt;
        const uint4* src = x + (size_t)t * H8;
        uint32_t mx = 0;  // max |bf16| bit pattern (orders like the magnitude)
        auto row_max = [&](const uint4& v) {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
        };
        if constexpr (NPL > 0) {
            uint4 v[NPL];
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int c = lane + 32 * i;
                v[i] = c < H8 ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < NPL; ++i) row_max(v[i]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
            const int sigma = row_f16_shift(mx);
            const float up = __uint_as_float((uint32_t)(127 + sigma) << 23);
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int c = lane + 32 * i;
                if (c < H8)
                    __stcs(dst + c, make_uint4(bf16x2_to_f16x2_scaled(v[i].x, up), bf16x2_to_f16x2_scaled(v[i].y, up),
                                               bf16x2_to_f16x2_scaled(v[i].z, up), bf16x2_to_f16x2_scaled(v[i].w, up)));
            }
            if (lane == 0) rscale[t] = __uint_as_float((uint32_t)(127 - sigma) << 23);
        } else {
#pragma unroll 4
            for (int c = lane; c < H8; c += 32) row_max(__ldg(src + c));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
            const int sigma = row_f16_shift(mx);
            const float up = __uint_as_float((uint32_t)(127 + sigma) << 23);
#pragma unroll 4
            for (int c = lane; c < H8; c += 32) {
                const uint4 v = __ldg(src + c);
                __stcs(dst + c, make_uint4(bf16x2_to_f16x2_scaled(v.x, up), bf16x2_to_f16x2_scaled(v.y, up),
                                           bf16x2_to_f16x2_scaled(v.z, up), bf16x2_to_f16x2_scaled(v.w, up)));
            }
            if (lane == 0) rscale[t] = __uint_as_float((uint32_t)(127 - sigma) << 23);
        }
    }
    pdl_end();
}

// out[t, m] = bf16(sum over j ascending of f[p] * (y16 * 2^-shift)), p =
// inv[t * Kt + j], for y staged by the down epilogues as f16 rows by sorted
// position ([cap][Hpad] halves, Hpad = H rounded up to 128) with a shift per
// (8 output rows, 32 positions) ([cap/32][Hpad/8] bytes).  8 consecutive m per
// thread, so one shift per slot: the slot's factor f[p] * 2^-shift is exact
// (a power of two times f[p]; the products it could push below the normal
// range are below 2^-110) and each term f[p] * y is rounded once (no fused
// multiply-add), then added in slot order, as moe_combine sums.  S slots'
// loads are in flight
// at a time: their index loads first, then their y loads.  S = 2 measured
// fastest on the 8192-token prefill (155 µs; 173 µs with 1, ~190 µs with 4,
// ~355 µs with 12, where the register count halves the resident warps).
template <int S>
__global__ void __launch_bounds__(256) combine_blocked_f16_kernel(const uint4* __restrict__ y16,
                                                                  const int8_t* __restrict__ shift,
                                                                  const int32_t* __restrict__ inv,
                                                                  const float* __restrict__ f, int T,
                                                                  int H, int Kt, int cap,
                                                                  uint4* __restrict__ out) {
    pdl_begin();
    const int H8 = H / 8, Hpad8 = (H + 127) / 128 * 16;
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < (size_t)T * H8) {
        const size_t t = i / H8;
        const int m8 = (int)(i % H8);
        float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j0 = 0; j0 < Kt; j0 += S) {
            int p[S];
            uint4 h[S];
            float c[S];
#pragma unroll
            for (int u = 0; u < S; ++u) p[u] = j0 + u < Kt ? __ldg(inv + t * Kt + j0 + u) : -1;
#pragma unroll
            for (int u = 0; u < S; ++u) {
                if ((unsigned)p[u] < (unsigned)cap) {
                    h[u] = __ldg(y16 + (size_t)p[u] * Hpad8 + m8);
                    const int sh = __ldg(shift + (size_t)(p[u] / 32) * Hpad8 + m8);
                    c[u] = (f ? __ldg(f + p[u]) : 1.0f) * __uint_as_float((uint32_t)(127 - sh) << 23);
                }
            }
#pragma unroll
            for (int u = 0; u < S; ++u) {
                if (j0 + u >= Kt) break;
                if ((unsigned)p[u] >= (unsigned)cap) {
                    flag_index_error();
                    continue;
                }
                const uint32_t hw[4] = {h[u].x, h[u].y, h[u].z, h[u].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 yy = __half22float2(*reinterpret_cast<const __half2*>(&hw[k]));
                    a[2 * k] = __fadd_rn(a[2 * k], __fmul_rn(yy.x, c[u]));
                    a[2 * k + 1] = __fadd_rn(a[2 * k + 1], __fmul_rn(yy.y, c[u]));
                }
            }
        }
        uint4 o;
        o.x = (uint32_t)f32_to_bf16_bits(a[0]) | ((uint32_t)f32_to_bf16_bits(a[1]) << 16);
        o.y = (uint32_t)f32_to_bf16_bits(a[2]) | ((uint32_t)f32_to_bf16_bits(a[3]) << 16);
        o.z = (uint32_t)f32_to_bf16_bits(a[4]) | ((uint32_t)f32_to_bf16_bits(a[5]) << 16);
        o.w = (uint32_t)f32_to_bf16_bits(a[6]) | ((uint32_t)f32_to_bf16_bits(a[7]) << 16);
        out[i] = o;
    }
    pdl_end();
}

}  // namespace

cudaError_t launch_combine_blocked_f16(const uint16_t* y16, const int8_t* shift, const int32_t* inv,
                                       const float* f, int T, int H, int Kt, int cap, uint16_t* out,
                                       cudaStream_t s) {
    const long long n = (long long)T * (H / 8);
    if (n <= 0) return cudaSuccess;
    const dim3 grid((unsigned)((n + 255) / 256)), block(256);
    const uint4* y = reinterpret_cast<const uint4*>(y16);
    uint4* o = reinterpret_cast<uint4*>(out);
    return launch_pdl(combine_blocked_f16_kernel<2>, grid, block, 0, s, y, shift, inv, f, T, H, Kt, cap, o);
}

cudaError_t launch_gather_rows_f16(const uint16_t* x, int H, const int32_t* sorted_pairs,
                                   const int32_t* num_tiles, int tile_m, int Kt, int cap,
                                   int num_pairs, uint16_t* xg, float* rscale, cudaStream_t s) {
    if (cap <= 0) return cudaSuccess;
    const int blocks = std::min((cap + 7) / 8, num_sms() * 8);
    // rows of up to 4096 values in registers (16 pieces of 16 bytes per lane)
    auto kernel = H / 8 <= 32 * 16 ? gather_rows_f16_kernel<16> : gather_rows_f16_kernel<0>;
    return launch_pdl(kernel, dim3(blocks), dim3(256), 0, s, reinterpret_cast<const uint4*>(x),
                      H / 8, sorted_pairs, num_tiles, tile_m, Kt, cap, num_pairs,
                      reinterpret_cast<uint4*>(xg), rscale);
}

bool prefill_tile_supported(int tile_m) {
    return tile_m == 32 || tile_m == 64 || tile_m == 128 || tile_m == 256;
}
bool prefill_shape_supported(int H, int I) { return H % 32 == 0 && I % 32 == 0; }
cudaError_t launch_prefill_gate_up(const GroupedGemm& g, cudaStream_t s) { return launch_mode<0>(g, s); }
cudaError_t launch_prefill_down(const GroupedGemm& g, cudaStream_t s) { return launch_mode<1>(g, s); }

cudaError_t read_device_error_prefill(int* flag, int clear) {
    int wait = 0, index = 0;
    cudaError_t err = cudaMemcpyFromSymbol(&wait, g_device_error, sizeof(int));
    if (err == cudaSuccess) err = cudaMemcpyFromSymbol(&index, g_index_error, sizeof(int));
    if (err != cudaSuccess) return err;
    *flag = (wait ? 1 : 0) | (index ? 2 : 0);
    if (!clear) return cudaSuccess;
    const int zero = 0;
    err = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    return err == cudaSuccess ? cudaMemcpyToSymbol(g_index_error, &zero, sizeof(int)) : err;
}

}  // namespace moe
